"""Host-side rule of the split state chains (no GPU): when a batch's long
documents run as composed segments, and how they are cut.

A long document's chain is split only when the batch is chain-bound: its
longest document has more than 32 chunks (of 64 tokens) and more than twice
the average chain length per resident chain CTA (two per SM: 304 on a
152-SM GB300).  Segments are the least multiple of 16 chunks whose square
covers the longest document.  The rule is compiled from the library's own
header into a small host program, and checked on the workloads it is meant
to separate: the 300M shape (32 chunks per row) and 16 rows of 8192 tokens
never split; the packed varlen row (one 128-chunk document among short ones)
and a lone long document do.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from kimi_delta_attention_bwd_gb300.inputs import WORKLOADS, make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kimi_delta_attention_bwd_gb300", "csrc")

PROGRAM = r'''
#include <cstdio>
#include "kda_internal.cuh"
int main() {
  int n_max, H, slots, n;
  long long total;
  // queries on stdin: "s n_max total H slots" -> seg_split; "l n_max" -> seg_len; "c n split len" -> seg_count
  char op;
  while (scanf(" %c", &op) == 1) {
    if (op == 's' && scanf("%d %lld %d %d", &n_max, &total, &H, &slots) == 4)
      printf("%d\n", kda::seg_split(n_max, total, H, slots) ? 1 : 0);
    else if (op == 'l' && scanf("%d", &n_max) == 1)
      printf("%d\n", kda::seg_len(n_max));
    else if (op == 'c' && scanf("%d %d %d", &n, &H, &slots) == 3)
      printf("%d\n", kda::seg_count(n, H != 0, slots));
  }
  return 0;
}
'''


@pytest.fixture(scope="module")
def rule(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("split_rule")
    src, exe = d / "rule.cu", d / "rule"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)

    def ask(*queries):
        out = subprocess.run([str(exe)], input="\n".join(" ".join(str(x) for x in q) for q in queries),
                             check=True, capture_output=True, text=True).stdout.split()
        return [int(x) for x in out]
    return ask


SLOTS = 2 * 152  # resident chain CTAs of a GB300


def chunks(lengths):
    return [(L + 63) // 64 for L in lengths]


def test_split_decisions_on_the_workloads(rule):
    varlen = np.diff(make_inputs(WORKLOADS[2], with_grad_inputs=False)["cu_seqlens"].numpy())
    cases = {
        "300M rows (16 x 2048, H 8)": (chunks([2048] * 16), 8, 0),
        "16 rows of 8192 tokens, H 8": (chunks([8192] * 16), 8, 0),
        "packed varlen row (1 x 32768, H 8)": (chunks(varlen), 8, 1),
        "4 rows of 8192 tokens, H 8": (chunks([8192] * 4), 8, 1),
        "one document of 33 chunks, H 2": (chunks([64 * 32 + 1]), 2, 1),
        "one document of 32 chunks, H 2": (chunks([64 * 32]), 2, 0),
    }
    got = rule(*[("s", max(c), sum(c), H, SLOTS) for c, H, _ in cases.values()])
    assert got == [want for _, _, want in cases.values()], dict(zip(cases, got))


def test_segment_lengths_and_counts(rule):
    # the least multiple of 16 whose square covers the longest document
    assert rule(("l", 33), ("l", 128), ("l", 256), ("l", 257), ("l", 301), ("l", 16384)) == [16, 16, 16, 32, 32, 128]
    # documents of at most 32 chunks stay whole; longer ones split into ceil(n / len) segments
    assert rule(("c", 32, 1, 16), ("c", 33, 1, 16), ("c", 128, 1, 16), ("c", 301, 1, 32), ("c", 128, 0, 16)) == \
        [1, 3, 8, 10, 1]
