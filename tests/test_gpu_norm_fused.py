"""KDA with the gated RMSNorm epilogue fused in (kda_fwd_norm_gate /
kda_bwd_norm_gate) against the KDA oracle composed with the norm oracle.

Forward: y = norm_gate(o) with o the KDA output.  Backward of
sum(y dy) + sum(h_final dh_final): the norm oracle's backward gives dO, dg and
dw; the KDA oracle's backward on dO gives the rest.  Both tensors that cross
between the two steps could be stored in the io dtype: o (the forward's
output, which the backward reads) and dO (an output, read back by the
per-chunk kernels).  The forward keeps o in fp32 for the backward, so the
norm oracle's backward takes the exact o; the KDA oracle's backward takes its
dO rounded to the io dtype, the tensor the fused path hands to its per-chunk
kernels.  The path rounds its own dO, which can sit one bf16 step from the
oracle's rounded dO; with bf16 io the token gradients' max-norm limit adds
twice the oracle's own sensitivity to that rounding (dO_rounding_tol), which
matters at the full 16 x 2048 size where some large dO element always lands on
a rounding boundary.  The rms limit stays.


bf16 at dk=32/dv=64 runs the fused chains (a cluster of two CTAs per document
and head exchanging row sums through distributed shared memory); other
shapes run kda_fwd plus the standalone norm kernels inside the same calls.
"""
import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_backward_norm_gate, kda_forward_norm_gate
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs, norm_gate_inputs
from oracle import norm_gate as ong
from _common import TOL_IO, compare, dO_rounding_tol, rel_max, rel_rms, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, seed, lengths)
    "rows_32_64": (custom(2, 300, 4, 32, 64, h0=True, dh_final=True), 31, None),
    "packed_one_token_and_empty_docs": (custom(1, 500, 2, 32, 64, h0=True, dh_final=True), 32, [1, 0, 130, 64, 305]),
    "scalar_gate": (custom(2, 200, 3, 32, 64, gate="scalar"), 33, None),
    "composed_fp32_128_128_packed": (custom(1, 300, 2, 128, 128, dtype="f32", h0=True, dh_final=True), 34,
                                     [100, 1, 199]),
    "composed_fp32": (custom(1, 192, 2, 32, 64, dtype="f32", h0=True, dh_final=True), 35, None),
    # the 300M layer shape the bench times (16 x 2048, H 8), with states
    "full_300M_16x2048": (custom(16, 2048, 8, 32, 64, h0=True, dh_final=True), 38, None),
    # a 41-chunk document packed with short ones, two heads: the forward chain runs it as composed
    # segments (the reverse chain, which forms dO itself, stays whole)
    "long_doc_split_forward": (custom(1, 64 * 40 + 17 + 150, 2, 32, 64, h0=True, dh_final=True), 39,
                               [64 * 40 + 17, 1, 0, 149]),
}


def _norm_inputs(w, seed):
    n = w.B * w.T * w.H
    x = norm_gate_inputs(n, w.dv, w.dtype, seed=seed + 500)
    shape = (w.B, w.T, w.H, w.dv)
    return x["g"].reshape(shape), x["w"], x["dy"].reshape(shape)


@pytest.mark.parametrize("name", list(CASES))
def test_fused_norm_matches_composed_oracles(name):
    w, seed, lens = CASES[name]
    inp = make_inputs(w, seed=seed, lengths=lens)
    g, wn, dy = _norm_inputs(w, seed)
    dev = "cuda"
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu_host = None if inp.get("cu_seqlens") is None else inp["cu_seqlens"].numpy()
    y, o, hf, ctx = kda_forward_norm_gate(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                          g.to(dev), wn.to(dev), scale=d["scale"], h0=d.get("h0"),
                                          cu_seqlens=d.get("cu_seqlens"), cu_seqlens_host=cu_host, want_o=True)
    gr = kda_backward_norm_gate(ctx, dy.to(dev), d.get("dh_final"))
    torch.cuda.synchronize()
    if name == "long_doc_split_forward":  # the forward chain splits, the reverse chain does not
        from kimi_delta_attention_bwd_gb300 import _lib
        _lib.prof_start()
        _, _, _, c2 = kda_forward_norm_gate(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                            g.to(dev), wn.to(dev), scale=d["scale"], h0=d.get("h0"),
                                            cu_seqlens=d.get("cu_seqlens"), cu_seqlens_host=cu_host, want_o=True)
        kda_backward_norm_gate(c2, dy.to(dev), d.get("dh_final"))
        torch.cuda.synchronize()
        launched = {k for k, v in _lib.prof_stop().items() if v[1]}
        assert "fwd_seg" in launched and "bwd_seg" not in launched, launched
        # offsets on the device only: the device plans the split on the grid of the most units any
        # offsets could give (the clusters past the last unit exit together); the same bits
        y3, o3, hf3, c3 = kda_forward_norm_gate(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                                                g.to(dev), wn.to(dev), scale=d["scale"], h0=d.get("h0"),
                                                cu_seqlens=d.get("cu_seqlens"), want_o=True)
        gr3 = kda_backward_norm_gate(c3, dy.to(dev), d.get("dh_final"))
        torch.cuda.synchronize()
        assert torch.equal(y3, y) and torch.equal(o3, o) and torch.equal(hf3, hf)
        for k2 in ("dO", "dg", "dw", "dq", "dk", "dv", "df", "db", "dA_log", "ddt_bias", "dh0"):
            assert torch.equal(gr3[k2], gr[k2]), k2
    N, H, dv = w.B * w.T, w.H, w.dv

    def host(t):
        return t.detach().double().cpu().numpy()

    ref = run_oracle(inp, False)
    g64, w64, dy64 = host(g).reshape(N, H, dv), host(wn), host(dy).reshape(N, H, dv)
    y_ref = ong.forward(ref["o"], g64, w64)
    dO_ref, dg_ref, dw_ref = ong.backward(ref["o"], g64, w64, dy64)
    bf = w.dtype == "bf16"
    errs = {}
    for n_, a, r in (("y", y, y_ref), ("dO", gr["dO"], dO_ref), ("dg", gr["dg"], dg_ref)):
        a = host(a).reshape(N, H, dv)
        assert np.isfinite(a).all(), n_
        errs[n_] = rel_max(a, r, bf16=bf)
        assert errs[n_] <= TOL_IO, (n_, errs)
        if bf:
            assert rel_rms(a, r) <= 5e-3, n_
    errs["dw"] = rel_max(host(gr["dw"]), dw_ref)
    assert errs["dw"] <= TOL_IO, errs
    # the KDA part: forward outputs, then the backward on dO as the fused path stores it
    inp_b = dict(inp)
    inp_b["dO"] = torch.from_numpy(dO_ref.reshape(w.B, w.T, H, dv)).to(inp["q"].dtype)
    refb = run_oracle(inp_b, True)
    tol_grad = None
    if bf:  # the path's dO is its own bf16 rounding: allow the oracle's sensitivity to one rounding
        refx = run_oracle(dict(inp, dO=torch.from_numpy(dO_ref.reshape(w.B, w.T, H, dv))), True)
        tol_grad = dO_rounding_tol(refb, refx)
        errs.update({"tol:" + k: v for k, v in tol_grad.items()})
    gpu = {"o": host(o).reshape(N, H, dv), "h_final": host(hf)}
    for k2 in ("dq", "dk", "dv", "df", "db"):
        t = host(gr[k2])
        gpu[k2] = t.reshape(N, H, *t.shape[3:]) if t.ndim == 4 else t.reshape(N, H)
    for k2 in ("dA_log", "ddt_bias", "dh0"):
        gpu[k2] = host(gr[k2])
    errs.update(compare(gpu, refb, True, bf16=bf, tol_grad=tol_grad))
    print(f"\n[fused norm] {name}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))


def test_fused_norm_without_o_and_deterministic():
    """Without saving, the fused forward need not write o and gives the same y
    bits; two fused backward calls give the same bits (fixed-order sums)."""
    w, seed, lens = CASES["rows_32_64"]
    inp = make_inputs(w, seed=seed, lengths=lens)
    g, wn, dy = _norm_inputs(w, seed)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    args = (d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], g.cuda(), wn.cuda())
    y1, o1, _, ctx = kda_forward_norm_gate(*args, scale=d["scale"], h0=d["h0"])
    y2, o2, _, _ = kda_forward_norm_gate(*args, scale=d["scale"], h0=d["h0"], save_for_backward=False)
    assert o1 is None and o2 is None and torch.equal(y1, y2)
    a = kda_backward_norm_gate(ctx, dy.cuda(), d["dh_final"])
    b = kda_backward_norm_gate(ctx, dy.cuda(), d["dh_final"])
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


def test_fused_norm_refuses_bf16_without_fused_kernels_and_foreign_workspaces():
    """bf16 at head shapes without the fused kernels is refused up front; a
    workspace saved by the plain forward is refused by the device."""
    from kimi_delta_attention_bwd_gb300 import KdaError, _lib, kda_device_status, kda_forward
    w = custom(1, 128, 2, 128, 128, h0=False)
    inp = make_inputs(w, seed=36)
    g, wn, dy = _norm_inputs(w, 36)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(KdaError) as ei:
        kda_forward_norm_gate(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], g.cuda(), wn.cuda())
    assert ei.value.status == -2
    w2, seed, _ = CASES["rows_32_64"]
    inp2 = make_inputs(w2, seed=seed)
    g2, wn2, dy2 = _norm_inputs(w2, seed)
    d2 = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp2.items()}
    ws = _lib.alloc_workspace(_lib.make_problem(w2.B, w2.T, w2.H, 32, 64, torch.bfloat16, d2["scale"]), 2)
    _, _, ctx = kda_forward(d2["q"], d2["k"], d2["v"], d2["f"], d2["b"], d2["A_log"], d2["dt_bias"],
                            scale=d2["scale"], h0=d2["h0"], workspace=ws)
    y, _, _, nctx = kda_forward_norm_gate(d2["q"], d2["k"], d2["v"], d2["f"], d2["b"], d2["A_log"], d2["dt_bias"],
                                          g2.cuda(), wn2.cuda(), scale=d2["scale"], h0=d2["h0"],
                                          save_for_backward=False)
    nctx.kda.workspace = ws  # saved by kda_forward, not by the fused forward
    nctx.saved = True
    kda_backward_norm_gate(nctx, dy2.cuda())
    assert kda_device_status(ws) == -5
