"""The allocation-free forward, kda_fwd_noalloc, called through the C ABI.

It exists for callers that cannot call cudaMalloc (a host program whose
device memory all belongs to its own pool, or a loop that cannot afford the
synchronisation an allocation may imply): its scratch is a fixed array inside
the library instead of a caller workspace.  Two calls in a row, on different
problems, must each match kda_fwd (which uses a caller workspace) within the
parity tolerances; a problem too big for the array is refused up front.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import _lib, kda_forward
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import TOL_IO, TOL_STATE, rel_fro, rel_max

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = _lib.load()
    fn = lib.kda_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(_lib.kda_problem)] + [ctypes.c_void_p] * 10 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(d, cu):
    B, T, H, dk = d["q"].shape
    dv = d["v"].shape[-1]
    n_docs = B if cu is None else cu.numel() - 1
    prob = _lib.make_problem(B, T, H, dk, dv, d["q"].dtype, d["scale"], cu, None)
    o = torch.empty(B, T, H, dv, dtype=d["q"].dtype, device="cuda")
    hf = torch.empty(n_docs, H, dk, dv, dtype=torch.float32, device="cuda")
    p = _lib._p
    st = _noalloc_fn()(ctypes.byref(prob), p(d["q"]), p(d["k"]), p(d["v"]), p(d["f"]), p(d["b"]), p(d["A_log"]),
                       p(d["dt_bias"]), p(d.get("h0")), p(o), p(hf), _lib._stream())
    return st, o, hf


@pytest.mark.parametrize("order", ["small_then_varlen", "varlen_then_small"])
def test_noalloc_matches_kda_fwd_on_consecutive_calls(order):
    cases = [
        (custom(2, 300, 4, 32, 64, dtype="bf16", h0=True), 21, None),
        (custom(1, 500, 2, 128, 128, dtype="bf16", h0=True), 22, [1, 0, 130, 64, 305]),
    ]
    if order == "varlen_then_small":
        cases = cases[::-1]
    for w, seed, lens in cases:
        inp = make_inputs(w, seed=seed, lengths=lens, with_grad_inputs=False)
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        cu = d.get("cu_seqlens")
        st, o, hf = _call_noalloc(d, cu)
        assert st == 0, _lib.strerror(st)
        o_ref, hf_ref, _ = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                       scale=d["scale"], h0=d["h0"], cu_seqlens=cu, save_for_backward=False)
        torch.cuda.synchronize()
        a, r = o.double().cpu().numpy(), o_ref.double().cpu().numpy()
        assert rel_max(a, r, bf16=True) <= TOL_IO
        assert rel_fro(hf.cpu().numpy(), hf_ref.cpu().numpy()) <= TOL_STATE


def test_noalloc_refuses_problems_beyond_its_array():
    # fp32 io takes the general kernels, whose forward scratch (fp32 intra-chunk
    # factors) is about 235 MB here
    big = _lib.make_problem(16, 2048, 8, 32, 64, torch.float32)
    assert _lib.kda_workspace_size(big, False) > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = _noalloc_fn()(ctypes.byref(big), *([fake] * 7), None, fake, None, None)
    assert st == -5
