"""Short causal convolution (kda_short_conv_fwd / _bwd) against its oracle:
dense and varlen (documents of every length, zero-length and one-token
documents, a document boundary inside and at the edge of a token tile),
bf16 and fp32, silu and no activation; bit-exact determinism of dw."""
import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_short_conv, kda_short_conv_backward
from kimi_delta_attention_bwd_gb300.inputs import cu_from_lengths, doc_lengths_docs600, short_conv_inputs
from oracle import short_conv as osc
from _common import TOL_IO, rel_max, rel_rms

pytestmark = pytest.mark.gpu


def _lengths_mixed(n):
    lens = [1, 0, 63, 64, 65, 1, 127, 128, 129, 3, 0, 255]
    lens.append(n - sum(lens))
    return lens


CASES = [
    ("dense bf16 C1024", 4096, 1024, "bf16", None, "silu"),
    ("varlen bf16 mixed", 1000, 256, "bf16", "mixed", "silu"),
    ("varlen fp32 docs600", 8192, 64, "f32", "docs600", "silu"),
    ("varlen bf16 no activation", 1000, 512, "bf16", "mixed", "none"),
]


@pytest.mark.parametrize("name,n,C,dt,docs,act", CASES, ids=[c[0] for c in CASES])
def test_short_conv_matches_oracle(name, n, C, dt, docs, act):
    inp = short_conv_inputs(n, C, dt, seed=11 + n + C)
    if docs == "mixed":
        cu = cu_from_lengths(_lengths_mixed(n))
    elif docs == "docs600":
        cu = cu_from_lengths(doc_lengths_docs600(n, np.random.RandomState(5)))
    else:
        cu = None
    d = {k: v.cuda() for k, v in inp.items()}
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    y = kda_short_conv(d["x"], d["w"], cu_d, activation=act)
    dx, dw = kda_short_conv_backward(d["x"], d["w"], d["dy"], cu_d, activation=act)
    torch.cuda.synchronize()
    f = {k: v.double().numpy() for k, v in inp.items()}
    ry = osc.forward(f["x"], f["w"], cu, activation=act)
    rdx, rdw = osc.backward(f["x"], f["w"], f["dy"], cu, activation=act)
    bf = dt == "bf16"
    for a, r in ((y, ry), (dx, rdx)):
        a = a.double().cpu().numpy()
        assert rel_max(a, r, bf16=bf) <= TOL_IO
        if bf:
            assert rel_rms(a, r) <= 5e-3
    assert rel_max(dw.cpu().numpy(), rdw, bf16=False) <= TOL_IO


def test_short_conv_backward_is_deterministic():
    inp = short_conv_inputs(3000, 256, "bf16", seed=2)
    d = {k: v.cuda() for k, v in inp.items()}
    a = kda_short_conv_backward(d["x"], d["w"], d["dy"])
    b = kda_short_conv_backward(d["x"], d["w"], d["dy"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
