"""The allocation-free forward, kda_fwd_noalloc, called through the C ABI.

It exists for callers that cannot call cudaMalloc (a host program whose
device memory all belongs to its own pool, or a loop that cannot afford the
synchronisation an allocation may imply): its scratch is a fixed array inside
the library instead of a caller workspace.  Two calls in a row, on different
problems, must each match kda_fwd (which uses a caller workspace) within the
parity tolerances; a problem too big for the array is refused up front.

At bf16, dk = 32, dv = 64 it runs its own single-kernel forward (one CTA per
document and head carries the state through the document's chunks), which no
other entry point uses; so that kernel is also checked against the CPU
oracle directly, on packed documents with one-token and empty ones, on the
scalar (GDN) gate, without an initial state and on gates whose 16-token
decay spans pass the 80-nat guard.  Offsets that exist only on the device
are checked by the device and reported by kda_noalloc_status().

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import _lib, kda_forward
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import TOL_IO, TOL_STATE, block_spans, compare, rel_fro, rel_max, run_oracle

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
    gate = _lib.KDA_GATE_SCALAR if d["f"].dim() == 3 else _lib.KDA_GATE_CHANNEL
    prob = _lib.make_problem(B, T, H, dk, dv, d["q"].dtype, d["scale"], cu, None, gate=gate)
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


CASES = {
    # name: (workload, seed, document lengths, gate mode)
    "packed_one_token_and_empty_docs": (custom(1, 500, 2, 32, 64, h0=True), 23, [1, 0, 130, 64, 305], None),
    "scalar_gate_no_h0": (custom(2, 300, 3, 32, 64, gate="scalar"), 24, None, None),
    "scalar_gate_packed": (custom(1, 260, 2, 32, 64, h0=True, gate="scalar"), 25, [64, 1, 0, 195], None),
    "spans_past_guard_packed": (custom(1, 400, 3, 32, 64, h0=True), 26, [1, 0, 70, 17, 64, 1, 200, 47], "fast"),
    "mixed_spans": (custom(2, 192, 2, 32, 64, h0=True), 27, None, "mixed"),
    "beta_one": (custom(2, 150, 2, 32, 64, h0=True), 28, None, "beta1"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_single_kernel_forward_matches_oracle(name):
    w, seed, lens, mode = CASES[name]
    inp = make_inputs(w, seed=seed, lengths=lens, with_grad_inputs=False)
    if mode == "fast":
        inp["A_log"].fill_(3.0)
        inp["f"].mul_(3.0).add_(1.0)
        assert (block_spans(inp) > 80.0).mean() > 0.5
    elif mode == "mixed":
        inp["A_log"].fill_(2.0)
        inp["f"].add_(2.0)
        assert 0.05 < (block_spans(inp) > 80.0).mean() < 0.95
    elif mode == "beta1":
        inp["b"].fill_(30.0)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu = d.get("cu_seqlens")
    st, o, hf = _call_noalloc(d, cu)
    assert st == 0, _lib.strerror(st)
    assert _lib.load().kda_noalloc_status(_lib._stream()) == 0
    B, T, H = inp["q"].shape[:3]
    gpu = {"o": o.double().cpu().numpy().reshape(B * T, H, -1), "h_final": hf.double().cpu().numpy()}
    assert np.isfinite(gpu["o"]).all() and np.isfinite(gpu["h_final"]).all()
    ref = run_oracle(inp, False)
    errs = compare(gpu, ref, False)
    print(f"\n[noalloc] {name}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))


def test_noalloc_reports_device_only_bad_offsets():
    """Offsets that exist only on the device are checked there: the call
    returns KDA_OK (nothing synchronises), writes nothing, and
    kda_noalloc_status() reports KDA_ERR_BAD_SEQLENS; the next valid call
    clears it."""
    B, T, H, dk, dv = 1, 128, 2, 32, 64
    dev = "cuda"
    q = torch.randn(B, T, H, dk, device=dev, dtype=torch.bfloat16)
    v = torch.randn(B, T, H, dv, device=dev, dtype=torch.bfloat16)
    b = torch.randn(B, T, H, device=dev, dtype=torch.bfloat16)
    A = torch.zeros(H, device=dev)
    dtb = torch.zeros(H, dk, device=dev)
    p = _lib._p
    lib = _lib.load()
    for cu_list, want in (([0, 100, 50, 128], -4), ([0, 50, 100, 128], 0)):
        cu = torch.tensor(cu_list, dtype=torch.int32, device=dev)
        prob = _lib.make_problem(B, T, H, dk, dv, torch.bfloat16, None, cu, None)
        o = torch.full((B, T, H, dv), 7.0, device=dev, dtype=torch.bfloat16)
        st = lib.kda_fwd_noalloc(ctypes.byref(prob), p(q), p(q), p(v), p(q), p(b), p(A), p(dtb), None, p(o), None,
                                 _lib._stream())
        assert st == 0
        assert lib.kda_noalloc_status(_lib._stream()) == want
        assert bool(torch.all(o == 7.0)) == (want != 0)
