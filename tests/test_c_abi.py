"""The boundary from C: a C99 program (tests/c/abi_host_checks.c) compiled
with gcc against include/kda.h and linked to the in-tree library, run on the
host.  It checks that the header is plain C, that the library links without
PyTorch, and the workspace sizing and host validation statuses (no GPU)."""
import os
import shutil
import subprocess

import pytest

from kimi_delta_attention_bwd_gb300 import _lib
from kimi_delta_attention_bwd_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_against_the_header_and_library(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    _lib.load()  # builds the library if it is missing
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(B.nvcc())), "include")
    exe = str(tmp_path / "abi_host_checks")
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-I", cuda_inc, os.path.join(HERE, "c", "abi_host_checks.c"), "-o", exe,
                           "-L", B.BUILD, "-lkda_gb300", f"-Wl,-rpath,{B.BUILD}"])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
