"""Shared helpers of the parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare them with the tolerances of the KDA spec."""
from __future__ import annotations

import numpy as np
import torch

from kimi_delta_attention_bwd_gb300.inputs import numpy_f64

# Tolerances: max|err| / rms(ref) <= 1e-2 for the outputs and every gradient,
# and relative Frobenius error <= 2e-3 for the fp32 states (final state and
# its gradient dS0).  For outputs stored in bf16 the max-norm applies to the
# computed value: the half-ulp rounding of the exact result to bf16, which no
# bf16-output implementation can avoid, is subtracted element-wise first
# (|err| - ulp_bf16(ref)/2, floored at 0).  Those outputs must also meet the
# pages' bf16 bar on the rms ratio, rms(err)/rms(ref) <= 5e-3, which includes
# the rounding.
TOL_IO = 1e-2
TOL_STATE = 2e-3
TOL_RMS_BF16 = 5e-3


def half_ulp_bf16(ref):
    """Half a unit in the last place of bf16 (8 significant bits) at |ref|."""
    _, e = np.frexp(np.abs(ref))
    return np.ldexp(1.0, e - 9) * (ref != 0)


def rel_max(got, ref, bf16=False):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    err = np.abs(got - ref)
    if bf16:
        err = np.maximum(err - half_ulp_bf16(ref), 0.0)
    if rms == 0.0:
        return float(err.max()) if got.size else 0.0
    return float(err.max() / rms)


def rel_rms(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    e = np.sqrt(np.mean((got - ref) ** 2)) if ref.size else 0.0
    return float(e / rms) if rms else float(e)


def rel_fro(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    n = np.linalg.norm(ref)
    if n == 0.0:
        return float(np.linalg.norm(got))
    return float(np.linalg.norm(got - ref) / n)


def to_dev(inp, device="cuda"):
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def run_gpu(inp, backward: bool, device="cuda"):
    """Runs kda_forward (and kda_backward) through the C ABI; returns float64
    numpy arrays in the flattened [Ntok, H, d] layout."""
    from kimi_delta_attention_bwd_gb300 import kda_forward, kda_backward
    d = to_dev(inp, device)
    cu_host = None if inp.get("cu_seqlens") is None else inp["cu_seqlens"].numpy()
    o, hf, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                             scale=d["scale"], h0=d.get("h0"), cu_seqlens=d.get("cu_seqlens"),
                             cu_seqlens_host=cu_host, save_for_backward=backward)
    B, T, H = inp["q"].shape[:3]
    res = {"o": o, "h_final": hf}
    if backward:
        g = kda_backward(ctx, d["dO"], d.get("dh_final"))
        res.update(g)
    torch.cuda.synchronize()
    out = {}
    for k, v in res.items():
        if v is None:
            continue
        v = v.detach().to(torch.float64).cpu().numpy()
        if k in ("o", "dq", "dk", "dv", "df", "db") and v.ndim >= 3:
            v = v.reshape(B * T, H, *v.shape[3:]) if v.ndim == 4 else v.reshape(B * T, H)
        out[k] = v
    return out


def run_oracle(inp, backward: bool, units=None, threads=None):
    """The oracle on the same inputs.  A scalar gate (f [.., H], dt_bias [H])
    is the per-channel gate with every channel equal: the oracle runs on f
    and dt_bias repeated over dk, and the gate gradients are summed over the
    channels (the chain rule of the broadcast)."""
    from oracle import oracle
    x = numpy_f64(inp)
    scalar = x["f"].ndim == x["q"].ndim - 1
    if scalar:
        dk = x["q"].shape[-1]
        x["f"] = np.repeat(x["f"][..., None], dk, axis=-1)
        x["dt_bias"] = np.repeat(x["dt_bias"][:, None], dk, axis=1)
    o, hf = oracle.forward(x, units=units, threads=threads)
    res = {"o": o, "h_final": hf}
    if backward:
        g = oracle.backward(x, x["dO"], x.get("dh_final"), units=units, threads=threads)
        if scalar:
            g["df"] = g["df"].sum(axis=-1)
            g["ddt_bias"] = g["ddt_bias"].sum(axis=-1)
        res.update(g)
    return res


def compare(gpu, ref, backward: bool, rows=None, states=None, params_heads=None, tol_io=TOL_IO,
            tol_state=TOL_STATE, bf16=True, tol_grad=None):
    """Returns {name: error} and asserts every error is within tolerance.
    rows/states: index arrays restricting the comparison to sampled units.
    tol_grad: {name: max-norm limit} for token gradients (dq, dk, dv, df,
    db) whose limit differs from tol_io (see dO_rounding_tol)."""
    errs = {}
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    sst = (lambda a: a) if states is None else (lambda a: a[states])
    io_names = ["o"] + (["dq", "dk", "dv", "df", "db"] if backward else [])
    for n in io_names:
        errs[n] = rel_max(sel(gpu[n]), sel(ref[n]), bf16)
        if bf16:
            errs[n + ":rms"] = rel_rms(sel(gpu[n]), sel(ref[n]))
    errs["h_final"] = rel_fro(sst(gpu["h_final"]), sst(ref["h_final"]))
    if backward:
        if "dh0" in gpu:
            errs["dh0"] = rel_fro(sst(gpu["dh0"]), sst(ref["dh0"]))
        ph = slice(None) if params_heads is None else params_heads
        errs["dA_log"] = rel_max(gpu["dA_log"][ph], ref["dA_log"][ph])
        errs["ddt_bias"] = rel_max(gpu["ddt_bias"][ph], ref["ddt_bias"][ph])
    bad = {}
    for n, e in errs.items():
        lim = tol_state if n in ("h_final", "dh0") else TOL_RMS_BF16 if n.endswith(":rms") else tol_io
        if tol_grad is not None and n in tol_grad:
            lim = tol_grad[n]
        if not (e <= lim):
            bad[n] = (e, lim)
    assert not bad, f"parity failures {bad}; all errors {errs}"
    return errs


GRAD_NAMES = ("dq", "dk", "dv", "df", "db")


def dO_rounding_tol(ref_rounded, ref_exact, names=GRAD_NAMES):
    """Per-gradient max-norm limits for a backward that takes a dO that a
    fused path computed itself and stored in bf16.

    The path's bf16 dO and the oracle's dO rounded to bf16 are two roundings
    of nearly equal values: they differ by one bf16 step wherever the two sit
    on opposite sides of a rounding boundary.  The backward is linear in dO,
    so the gradients move by the backward of that one-step difference.  Its
    scale is measured on the oracle alone: the oracle's backward on its exact
    dO (ref_exact) against the same on that dO rounded (ref_rounded) is the
    response to a perturbation of up to half a step on every element; twice
    that is taken as the response to a full step.  Returns {name: TOL_IO plus
    twice that gradient's move} (relative max-norm, as rel_max).  The rms
    limit is unchanged."""
    return {n: TOL_IO + 2.0 * rel_max(ref_rounded[n], ref_exact[n]) for n in names}


def block_spans(inp, chunk=64, block=16):
    """Decay span in nats of every 16-token block of every 64-token chunk
    (chunks restart at each document): for channel i, minus the sum of the
    log-decays g of the block's rows after its first, i.e. G_first - G_last
    of the in-chunk cumulative gate.  Returns the per-block maximum over the
    channels and heads.  The tensor-core kernels evaluate a diagonal block
    pairwise and exactly when this exceeds 80."""
    x = numpy_f64(inp)
    f, dtb, A = x["f"], x["dt_bias"], x["A_log"]
    N, H = x["q"].shape[:2]
    if f.ndim == 2:  # scalar gate: one value per token and head
        f = f[..., None]
        dtb = dtb[:, None]
    g = -np.exp(A)[None, :, None] * np.logaddexp(0.0, f + dtb[None])
    cu = x["cu_seqlens"]
    spans = []
    for d in range(len(cu) - 1):
        for c0 in range(int(cu[d]), int(cu[d + 1]), chunk):
            c1 = min(c0 + chunk, int(cu[d + 1]))
            for b0 in range(c0, c1, block):
                b1 = min(b0 + block, c1)
                spans.append(float(-g[b0 + 1:b1].sum(axis=0).min()) if b1 - b0 > 1 else 0.0)
    return np.array(spans)
