"""The layer with the short convolution fused into the per-chunk kernels
(kda_fwd_conv / kda_bwd_conv) against the oracles composed: the convolution
oracle (oracle/short_conv.py), the KDA oracle on its exact outputs, and with
g given the gated-norm oracle; the backward chains the three oracles'
backwards in reverse.

As in the fused-norm test, the one tensor the fused backward stores in the io
dtype between the steps, dO (with the norm), enters the KDA oracle's backward
rounded to that dtype; the gradients downstream of it (dx, df, db) then take
the max-norm limit widened by the oracle's own sensitivity to that rounding
(dO_rounding_tol).  q, k, v are never rounded: the kernels apply the
convolution to the rows they load and keep its fp32 outputs, so the KDA
oracle takes the convolution oracle's exact outputs.

Cases: rows, packed documents with one-token and empty ones (the window and
the state reset at each document), the scalar gate, gates whose 16-token
spans pass the 80-nat guard (the exact fallback recomputes q and k through
the convolution), the norm, and a long packed document on which both state
chains run split into composed segments.
"""
import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_backward_conv, kda_forward_conv
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs, norm_gate_inputs, short_conv_inputs
from oracle import norm_gate as ong
from oracle import short_conv as osc
from _common import TOL_IO, TOL_STATE, block_spans, dO_rounding_tol, rel_fro, rel_max, rel_rms, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, seed, lengths, norm, gate mode)
    "rows": (custom(2, 300, 4, 32, 64, h0=True, dh_final=True), 41, None, False, None),
    "packed_docs_norm": (custom(1, 500, 2, 32, 64, h0=True, dh_final=True), 42, [1, 0, 130, 2, 64, 303], True, None),
    "scalar_gate_norm": (custom(2, 200, 3, 32, 64, gate="scalar"), 43, None, True, None),
    "wide_spans_packed": (custom(1, 400, 2, 32, 64, h0=True, dh_final=True), 44, [1, 0, 70, 17, 64, 1, 200, 47], False,
                          "fast"),
    # the 300M layer shape the bench times (16 x 2048, H 8), with the norm and states
    "full_300M_16x2048_norm": (custom(16, 2048, 8, 32, 64, h0=True, dh_final=True), 45, None, True, None),
    # a 41-chunk document packed with a short one, few heads: without the norm both state chains
    # run split into composed segments (the fused-norm chains never split)
    "long_doc_split_chains": (custom(1, 64 * 40 + 17 + 13, 2, 32, 64, h0=True, dh_final=True), 46,
                              [64 * 40 + 17, 13], False, None),
    # the same with the norm: the forward chain (fused norm) splits, the reverse chain stays whole
    "long_doc_split_norm": (custom(1, 64 * 36 + 40 + 1, 2, 32, 64, h0=True, dh_final=True), 47,
                            [64 * 36 + 40, 1], True, None),
}


def _inputs(name):
    w, seed, lens, norm, mode = CASES[name]
    inp = make_inputs(w, seed=seed, lengths=lens)
    if mode == "fast":
        inp["A_log"].fill_(3.0)
        inp["f"].mul_(3.0).add_(1.0)
    C = w.H * (2 * w.dk + w.dv)
    cv = short_conv_inputs(w.B * w.T, C, "bf16", seed=seed + 700)
    x = cv["x"].reshape(w.B, w.T, C)
    g = wn = None
    if norm:
        ng = norm_gate_inputs(w.B * w.T * w.H, w.dv, "bf16", seed=seed + 800)
        g, wn = ng["g"].reshape(w.B, w.T, w.H, w.dv), ng["w"]
    dy = torch.randn(w.B, w.T, w.H, w.dv, generator=torch.Generator().manual_seed(seed + 900)).to(torch.bfloat16)
    return w, inp, x, cv["w"], g, wn, dy


@pytest.mark.parametrize("name", list(CASES))
def test_fused_conv_layer_matches_composed_oracles(name):
    w, inp, x, cw, g, wn, dy = _inputs(name)
    if CASES[name][4] == "fast":
        assert (block_spans(inp) > 80.0).mean() > 0.5  # spans computed from f alone: the convolution does not touch f
    dev = "cuda"
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu_host = None if inp.get("cu_seqlens") is None else inp["cu_seqlens"].numpy()
    out, hf, ctx = kda_forward_conv(x.to(dev), cw.to(dev), d["f"], d["b"], d["A_log"], d["dt_bias"], w.dk, w.dv,
                                    g=None if g is None else g.to(dev), w=None if wn is None else wn.to(dev),
                                    scale=d["scale"], h0=d.get("h0"), cu_seqlens=d.get("cu_seqlens"),
                                    cu_seqlens_host=cu_host)
    gr = kda_backward_conv(ctx, dy.to(dev), d.get("dh_final"))
    torch.cuda.synchronize()
    if name.startswith("long_doc_split"):  # the case does split (the reverse chain only without the norm)
        from kimi_delta_attention_bwd_gb300 import _lib
        _lib.prof_start()
        _, _, c2 = kda_forward_conv(x.to(dev), cw.to(dev), d["f"], d["b"], d["A_log"], d["dt_bias"], w.dk, w.dv,
                                    g=None if g is None else g.to(dev), w=None if wn is None else wn.to(dev),
                                    scale=d["scale"], h0=d.get("h0"), cu_seqlens=d.get("cu_seqlens"),
                                    cu_seqlens_host=cu_host)
        kda_backward_conv(c2, dy.to(dev), d.get("dh_final"))
        torch.cuda.synchronize()
        launched = {k for k, v in _lib.prof_stop().items() if v[1]}
        assert "fwd_seg" in launched and ("bwd_seg" in launched) == (g is None), launched
    N, H, dk, dv = w.B * w.T, w.H, w.dk, w.dv
    C = H * (2 * dk + dv)

    def host(t):
        return t.detach().double().cpu().numpy()

    cu = (np.arange(w.B + 1) * w.T) if inp.get("cu_seqlens") is None else inp["cu_seqlens"].numpy()
    x64, cw64 = host(x).reshape(N, C), host(cw)
    qkv = osc.forward(x64, cw64, cu)  # the convolution oracle, exact
    shp = lambda a, n: torch.from_numpy(np.ascontiguousarray(a.reshape(w.B, w.T, H, n)))
    inp_k = dict(inp, q=shp(qkv[:, :H * dk], dk), k=shp(qkv[:, H * dk:2 * H * dk], dk), v=shp(qkv[:, 2 * H * dk:], dv))
    ref = run_oracle(inp_k, False)
    errs = {}
    dy64 = host(dy).reshape(N, H, dv)
    if g is not None:
        g64, w64 = host(g).reshape(N, H, dv), host(wn)
        y_ref = ong.forward(ref["o"], g64, w64)
        dO_ref, dg_ref, dw_ref = ong.backward(ref["o"], g64, w64, dy64)
        for n_, a, r in (("y", out, y_ref), ("dO", gr["dO"], dO_ref), ("dg", gr["dg"], dg_ref)):
            errs[n_] = rel_max(host(a).reshape(N, H, dv), r, bf16=True)
            assert errs[n_] <= TOL_IO, (n_, errs)
        errs["dw"] = rel_max(host(gr["dw"]), dw_ref)
        assert errs["dw"] <= TOL_IO, errs
        dO_kda = torch.from_numpy(dO_ref.reshape(w.B, w.T, H, dv)).to(torch.bfloat16)
        dO_exact = torch.from_numpy(dO_ref.reshape(w.B, w.T, H, dv))
    else:
        errs["o"] = rel_max(host(out).reshape(N, H, dv), ref["o"], bf16=True)
        assert errs["o"] <= TOL_IO and rel_rms(host(out).reshape(N, H, dv), ref["o"]) <= 5e-3, errs
        dO_kda = dy
    inp_b = dict(inp_k, dO=dO_kda)
    refb = run_oracle(inp_b, True)

    def conv_back(r):
        dqkv = np.concatenate([r["dq"].reshape(N, -1), r["dk"].reshape(N, -1), r["dv"].reshape(N, -1)], axis=1)
        return osc.backward(x64, cw64, dqkv, cu)
    dx_ref, dcw_ref = conv_back(refb)
    refb["dx"] = dx_ref
    tol_grad = {"dx": TOL_IO, "df": TOL_IO, "db": TOL_IO}
    if g is not None:  # the path's dO is its own bf16 rounding: allow the oracle's sensitivity to one rounding
        refx = run_oracle(dict(inp_k, dO=dO_exact), True)
        refx["dx"] = conv_back(refx)[0]
        tol_grad = dO_rounding_tol(refb, refx, ("dx", "df", "db"))
        errs.update({"tol:" + k: v for k, v in tol_grad.items()})
    errs["dx"] = rel_max(host(gr["dx"]).reshape(N, C), dx_ref, bf16=True)
    errs["dx:rms"] = rel_rms(host(gr["dx"]).reshape(N, C), dx_ref)
    errs["dconv_w"] = rel_max(host(gr["dconv_w"]), dcw_ref)
    assert errs["dx"] <= tol_grad["dx"] and errs["dx:rms"] <= 5e-3 and errs["dconv_w"] <= TOL_IO, errs
    errs["h_final"] = rel_fro(host(hf), ref["h_final"])
    errs["dh0"] = rel_fro(host(gr["dh0"]), refb["dh0"])
    assert errs["h_final"] <= TOL_STATE and errs["dh0"] <= TOL_STATE, errs
    for k2 in ("df", "db"):
        t = host(gr[k2])
        t = t.reshape(N, H, *t.shape[3:]) if t.ndim == 4 else t.reshape(N, H)
        errs[k2] = rel_max(t, refb[k2], bf16=True)
        errs[k2 + ":rms"] = rel_rms(t, refb[k2])
        assert errs[k2] <= tol_grad[k2] and errs[k2 + ":rms"] <= 5e-3, errs
    for k2 in ("dA_log", "ddt_bias"):
        errs[k2] = rel_max(host(gr[k2]), refb[k2])
        assert errs[k2] <= TOL_IO, errs
    print(f"\n[fused conv] {name}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))


def test_fused_conv_deterministic_and_reset_at_documents():
    """Two backward calls give the same bits; a packed row equals the separate
    per-document runs bitwise (the window and the state reset at each start)."""
    w, inp, x, cw, g, wn, dy = _inputs("packed_docs_norm")
    dev = "cuda"
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    args = dict(g=g.to(dev), w=wn.to(dev), scale=d["scale"])
    out, hf, ctx = kda_forward_conv(x.to(dev), cw.to(dev), d["f"], d["b"], d["A_log"], d["dt_bias"], w.dk, w.dv,
                                    h0=d["h0"], cu_seqlens=d["cu_seqlens"], **args)
    a = kda_backward_conv(ctx, dy.to(dev), d["dh_final"])
    b = kda_backward_conv(ctx, dy.to(dev), d["dh_final"])
    for k in a:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k
    cu = inp["cu_seqlens"].numpy()
    for s in range(len(cu) - 1):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        if t1 == t0:
            continue
        sl = lambda t: t[:, t0:t1].clone()  # a fresh, aligned allocation
        o1, h1, c1 = kda_forward_conv(sl(x).to(dev), cw.to(dev), sl(d["f"]), sl(d["b"]), d["A_log"], d["dt_bias"],
                                      w.dk, w.dv, h0=d["h0"][s:s + 1].contiguous(), g=sl(args["g"]), w=args["w"],
                                      scale=d["scale"])
        g1 = kda_backward_conv(c1, sl(dy.to(dev)), d["dh_final"][s:s + 1].contiguous())
        assert torch.equal(o1, out[:, t0:t1]), s
        assert torch.equal(h1[0], hf[s]), s
        assert torch.equal(g1["dx"], a["dx"][:, t0:t1]), s
