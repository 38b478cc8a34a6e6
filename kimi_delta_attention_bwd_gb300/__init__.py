"""Kimi Delta Attention (KDA) chunked gated delta rule on GB300 (sm_103a).

Public API (PyTorch tensors on the CUDA device; the work runs in
libkda_gb300.so through its C ABI, include/kda.h):

  o, h_final, ctx = kda_forward(q, k, v, f, b, A_log, dt_bias, ...)
  grads = kda_backward(ctx, dO, dh_final=None)
  o = kda_decode_step(q, k, v, f, b, A_log, dt_bias, state)   # one token, state in place
  qkv = kda_short_conv(qkv_raw, conv_w, cu_seqlens)            # short causal conv (k=4) + silu
  y = kda_norm_gate(o, gate, weight)                           # gated RMSNorm epilogue
  y, o, h_final, ctx = kda_forward_norm_gate(q, ..., gate, weight)  # KDA with the epilogue fused
  grads = kda_backward_norm_gate(ctx, dy)                      # dq .. dh0, dO, dgate, dweight
  out, h_final, ctx = kda_forward_conv(x, conv_w, f, ...)      # short conv -> KDA (-> gated norm), fused
  grads = kda_backward_conv(ctx, dy)                           # dx, dconv_w, df, db, ...
  do, dgate, dweight = kda_norm_gate_backward(o, gate, weight, dy)
  o = kda_attention(q, k, v, f, b, A_log, dt_bias)             # the same as a torch.autograd op
  x = short_conv(x_raw, conv_w); y = gated_norm(o, gate, weight)  # likewise

Layouts: q, k, f [B, T, H, dk]; v [B, T, H, dv]; b [B, T, H] (bf16 or fp32);
A_log [H], dt_bias [H, dk] fp32 (scalar-gated variant: f [B, T, H], dt_bias [H]); optional cu_seqlens int32 [n_docs + 1] over
the flattened B*T tokens; states [n_docs, H, dk, dv] fp32.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib
from ._lib import KdaError, kda_device_status, kda_strerror_text  # noqa: F401

__all__ = ["kda_forward", "kda_backward", "kda_forward_norm_gate", "kda_backward_norm_gate", "kda_forward_conv",
           "kda_backward_conv", "kda_decode_step", "kda_norm_gate", "kda_norm_gate_backward",
           "kda_short_conv", "kda_short_conv_backward", "KdaContext", "KdaError", "kda_device_status",
           "kda_attention", "short_conv", "gated_norm"]


@dataclass
class KdaContext:
    problem: object
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    f: torch.Tensor
    b: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    h0: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    cu_seqlens_host: object
    workspace: torch.Tensor
    n_docs: int


def _check(t, name, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _shape(t, name, shape):
    """Shapes are checked before anything is launched: the C ABI sees only
    pointers, so a tensor smaller than its declared layout would be read out
    of bounds."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _dims(t, name, n):
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")


def _gate_of(f, dt_bias, qshape):
    """Gate mode from the shapes: f with q's shape (dt_bias [H, dk]) is KDA's
    per-channel gate; f without the dk axis (dt_bias [H]) is the scalar gate."""
    *lead, H, dk = qshape
    if tuple(f.shape) == tuple(qshape):
        if tuple(dt_bias.shape) != (H, dk):
            raise ValueError(f"dt_bias must be {(H, dk)} for a per-channel gate")
        return _lib.KDA_GATE_CHANNEL
    if tuple(f.shape) == tuple(lead) + (H,):
        if tuple(dt_bias.shape) != (H,):
            raise ValueError(f"dt_bias must be {(H,)} for a scalar gate")
        return _lib.KDA_GATE_SCALAR
    raise ValueError(f"f must be {tuple(qshape)} (per-channel gate) or {tuple(lead) + (H,)} (scalar gate)")


def kda_forward(q, k, v, f, b, A_log, dt_bias, scale: Optional[float] = None, h0=None,
                cu_seqlens=None, cu_seqlens_host=None, save_for_backward: bool = True,
                workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                want_final_state: bool = True, final_state: Optional[torch.Tensor] = None):
    """Forward pass.  Returns (o, h_final or None, ctx); ctx feeds kda_backward
    when save_for_backward is set.  out / final_state: optional preallocated
    outputs (final_state is written when want_final_state is set)."""
    _dims(q, "q", 4)
    _dims(v, "v", 4)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _shape(k, "k", q.shape)
    _shape(v, "v", (B, T, H, dv))
    _shape(b, "b", (B, T, H))
    _shape(A_log, "A_log", (H,))
    gate = _gate_of(f, dt_bias, (B, T, H, dk))
    if cu_seqlens is not None:
        _dims(cu_seqlens, "cu_seqlens", 1)
        if cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must hold at least two offsets")
    n_docs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if h0 is not None:
        _shape(h0, "h0", (n_docs, H, dk, dv))
    if out is not None:
        _shape(out, "out", (B, T, H, dv))
    if final_state is not None:
        _shape(final_state, "final_state", (n_docs, H, dk, dv))
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (f, "f"), (b, "b")):
        _check(t, n, q.dtype)
    _check(A_log, "A_log", torch.float32)
    _check(dt_bias, "dt_bias", torch.float32)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32)
    if h0 is not None:
        _check(h0, "h0", torch.float32)
    if out is not None:
        _check(out, "out", q.dtype)
    if final_state is not None:
        _check(final_state, "final_state", torch.float32)
    prob = _lib.make_problem(B, T, H, dk, dv, q.dtype, scale, cu_seqlens, cu_seqlens_host, gate)
    if workspace is None:
        workspace = _lib.alloc_workspace(prob, save_for_backward, q.device)
    o = out if out is not None else torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    hf = None
    if want_final_state:
        hf = final_state if final_state is not None else torch.empty(n_docs, H, dk, dv, dtype=torch.float32,
                                                                     device=q.device)
    _lib.kda_fwd(prob, q, k, v, f, b, A_log, dt_bias, h0, o, hf, save_for_backward, workspace)
    ctx = KdaContext(prob, q, k, v, f, b, A_log, dt_bias, h0, cu_seqlens, cu_seqlens_host, workspace, n_docs)
    return o, hf, ctx


def kda_backward(ctx: KdaContext, dO, dh_final=None, want_dh0: bool = True, grads: Optional[dict] = None):
    """Backward of sum(o * dO) + sum(h_final * dh_final).  Returns a dict with
    dq, dk, dv, df, db (io dtype), dA_log, ddt_bias, dh0 (fp32)."""
    q = ctx.q
    B, T, H, dk = q.shape
    dv = ctx.v.shape[-1]
    _shape(dO, "dO", (B, T, H, dv))
    if dh_final is not None:
        _shape(dh_final, "dh_final", (ctx.n_docs, H, dk, dv))
    outs = ()
    if grads is not None:  # caller-supplied outputs: the shapes and dtypes of what they receive
        outs = [(n, like.shape, like.dtype) for n, like in (("dq", q), ("dk", ctx.k), ("dv", ctx.v), ("df", ctx.f),
                                                            ("db", ctx.b), ("dA_log", ctx.A_log),
                                                            ("ddt_bias", ctx.dt_bias))]
        if grads.get("dh0") is not None:
            outs.append(("dh0", (ctx.n_docs, H, dk, dv), torch.float32))
        for n, shape, _ in outs:
            _shape(grads[n], n, shape)
    _check(dO, "dO", q.dtype)
    if dh_final is not None:
        _check(dh_final, "dh_final", torch.float32)
    for n, _, dtype in outs:
        _check(grads[n], n, dtype)
    if grads is None:
        grads = {
            "dq": torch.empty_like(q), "dk": torch.empty_like(ctx.k), "dv": torch.empty_like(ctx.v),
            "df": torch.empty_like(ctx.f), "db": torch.empty_like(ctx.b),
            "dA_log": torch.empty(H, dtype=torch.float32, device=q.device),
            "ddt_bias": torch.empty_like(ctx.dt_bias),
            "dh0": torch.empty(ctx.n_docs, H, dk, dv, dtype=torch.float32, device=q.device) if want_dh0 else None,
        }
    _lib.kda_bwd(ctx.problem, ctx.q, ctx.k, ctx.v, ctx.f, ctx.b, ctx.A_log, ctx.dt_bias, ctx.h0, dO, dh_final,
                 grads["dq"], grads["dk"], grads["dv"], grads["df"], grads["db"], grads["dA_log"],
                 grads["ddt_bias"], grads.get("dh0"), ctx.workspace)
    return grads


@dataclass
class KdaNormContext:
    """What kda_backward_norm_gate needs from kda_forward_norm_gate (the
    workspace inside kda holds o in fp32)."""
    kda: KdaContext
    g: torch.Tensor
    w: torch.Tensor
    eps: float
    saved: bool


def kda_forward_norm_gate(q, k, v, f, b, A_log, dt_bias, g, w, eps: Optional[float] = None,
                          scale: Optional[float] = None, h0=None, cu_seqlens=None, cu_seqlens_host=None,
                          save_for_backward: bool = True, workspace: Optional[torch.Tensor] = None,
                          want_final_state: bool = True, want_o: bool = False):
    """KDA forward with the gated RMSNorm epilogue y = o r w sigmoid(g) fused in
    (g [B, T, H, dv] in the io dtype, w [dv] fp32).  Returns (y, o or None,
    h_final or None, ctx); o (the pre-norm output, io dtype) is returned when
    asked for (want_o), or when it is the intermediate of the composed path
    (head shapes other than 32/64, fp32 io, without saving)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    _shape(g, "g", (B, T, H, dv))
    _shape(w, "w", (dv,))
    _check(g, "g", q.dtype)
    _check(w, "w", torch.float32)
    _shape(k, "k", q.shape)
    _shape(v, "v", (B, T, H, dv))
    _shape(b, "b", (B, T, H))
    _shape(A_log, "A_log", (H,))
    gate = _gate_of(f, dt_bias, (B, T, H, dk))
    n_docs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if h0 is not None:
        _shape(h0, "h0", (n_docs, H, dk, dv))
        _check(h0, "h0", torch.float32)
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (f, "f"), (b, "b")):
        _check(t, n, q.dtype)
    _check(A_log, "A_log", torch.float32)
    _check(dt_bias, "dt_bias", torch.float32)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32)
    prob = _lib.make_problem(B, T, H, dk, dv, q.dtype, scale, cu_seqlens, cu_seqlens_host, gate)
    if workspace is None:
        workspace = _lib.alloc_workspace(prob, 2 if save_for_backward else 0, q.device)
    y = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    composed_intermediate = not save_for_backward and not (q.dtype == torch.bfloat16 and (dk, dv) == (32, 64))
    o = torch.empty_like(y) if (want_o or composed_intermediate) else None
    hf = torch.empty(n_docs, H, dk, dv, dtype=torch.float32, device=q.device) if want_final_state else None
    _lib.kda_fwd_norm_gate(prob, q, k, v, f, b, A_log, dt_bias, h0, g, w, eps, o, y, hf, save_for_backward,
                           workspace)
    ctx = KdaNormContext(KdaContext(prob, q, k, v, f, b, A_log, dt_bias, h0, cu_seqlens, cu_seqlens_host, workspace,
                                    n_docs), g, w, float(eps or 0.0), bool(save_for_backward))
    return y, o, hf, ctx


def kda_backward_norm_gate(ctx: KdaNormContext, dy, dh_final=None, want_dh0: bool = True):
    """Backward of sum(y * dy) + sum(h_final * dh_final) through the fused
    epilogue.  Returns kda_backward's gradients plus dO (of the pre-norm
    output), dg and dw."""
    c = ctx.kda
    q = c.q
    B, T, H, dk = q.shape
    dv = c.v.shape[-1]
    if not ctx.saved:
        raise ValueError("the forward saved nothing: call kda_forward_norm_gate with save_for_backward=True")
    _shape(dy, "dy", (B, T, H, dv))
    _check(dy, "dy", q.dtype)
    if dh_final is not None:
        _shape(dh_final, "dh_final", (c.n_docs, H, dk, dv))
        _check(dh_final, "dh_final", torch.float32)
    gr = {
        "dq": torch.empty_like(q), "dk": torch.empty_like(c.k), "dv": torch.empty_like(c.v),
        "df": torch.empty_like(c.f), "db": torch.empty_like(c.b),
        "dA_log": torch.empty(H, dtype=torch.float32, device=q.device), "ddt_bias": torch.empty_like(c.dt_bias),
        "dh0": torch.empty(c.n_docs, H, dk, dv, dtype=torch.float32, device=q.device) if want_dh0 else None,
        "dO": torch.empty_like(dy), "dg": torch.empty_like(dy),
        "dw": torch.empty(dv, dtype=torch.float32, device=q.device),
    }
    _lib.kda_bwd_norm_gate(c.problem, c.q, c.k, c.v, c.f, c.b, c.A_log, c.dt_bias, c.h0, ctx.g, ctx.w, ctx.eps,
                           dy, dh_final, gr["dO"], gr["dg"], gr["dw"], gr["dq"], gr["dk"], gr["dv"], gr["df"],
                           gr["db"], gr["dA_log"], gr["ddt_bias"], gr["dh0"], c.workspace)
    return gr


@dataclass
class KdaConvContext:
    """What kda_backward_conv needs from kda_forward_conv."""
    problem: object
    x: torch.Tensor
    conv_w: torch.Tensor
    f: torch.Tensor
    b: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    h0: Optional[torch.Tensor]
    g: Optional[torch.Tensor]
    w: Optional[torch.Tensor]
    eps: float
    cu_seqlens: Optional[torch.Tensor]
    cu_seqlens_host: object
    workspace: torch.Tensor
    n_docs: int
    dk: int
    dv: int
    saved: bool


def kda_forward_conv(x, conv_w, f, b, A_log, dt_bias, dk: int, dv: int, g=None, w=None, eps: Optional[float] = None,
                     scale: Optional[float] = None, h0=None, cu_seqlens=None, cu_seqlens_host=None,
                     save_for_backward: bool = True, workspace: Optional[torch.Tensor] = None,
                     want_final_state: bool = True):
    """The layer in one call: q | k | v = silu(conv4(x)) per document, KDA, and
    (g, w given) the gated RMSNorm.  x [B, T, H (2 dk + dv)] (q channels, then
    k, then v), conv_w [H (2 dk + dv), 4] fp32.  Returns (out, h_final or None,
    ctx): out is y with the norm, o without."""
    _dims(x, "x", 3)
    B, T, Cx = x.shape
    H = A_log.shape[0]
    if Cx != H * (2 * dk + dv):
        raise ValueError(f"x has {Cx} channels; H (2 dk + dv) = {H * (2 * dk + dv)}")
    _shape(conv_w, "conv_w", (Cx, 4))
    _shape(b, "b", (B, T, H))
    _shape(A_log, "A_log", (H,))
    gate = _gate_of(f, dt_bias, (B, T, H, dk))
    n_docs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if h0 is not None:
        _shape(h0, "h0", (n_docs, H, dk, dv))
        _check(h0, "h0", torch.float32)
    for t, n in ((x, "x"), (f, "f"), (b, "b")):
        _check(t, n, x.dtype)
    _check(conv_w, "conv_w", torch.float32)
    _check(A_log, "A_log", torch.float32)
    _check(dt_bias, "dt_bias", torch.float32)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32)
    if g is not None:
        _shape(g, "g", (B, T, H, dv))
        _shape(w, "w", (dv,))
        _check(g, "g", x.dtype)
        _check(w, "w", torch.float32)
    prob = _lib.make_problem(B, T, H, dk, dv, x.dtype, scale, cu_seqlens, cu_seqlens_host, gate)
    if workspace is None:
        workspace = _lib.alloc_workspace(prob, 3 if save_for_backward else 0, x.device)
    out = torch.empty(B, T, H, dv, dtype=x.dtype, device=x.device)
    o, y = (out, None) if g is None else (None, out)
    hf = torch.empty(n_docs, H, dk, dv, dtype=torch.float32, device=x.device) if want_final_state else None
    _lib.kda_fwd_conv(prob, x, conv_w, f, b, A_log, dt_bias, h0, g, w, eps, o, y, hf, save_for_backward, workspace)
    ctx = KdaConvContext(prob, x, conv_w, f, b, A_log, dt_bias, h0, g, w, float(eps or 0.0), cu_seqlens,
                         cu_seqlens_host, workspace, n_docs, dk, dv, bool(save_for_backward))
    return out, hf, ctx


def kda_backward_conv(ctx: KdaConvContext, dy, dh_final=None, want_dh0: bool = True):
    """Backward of the layer: dy is the gradient of its output (y with the
    norm, o without).  Returns dx, dconv_w, df, db, dA_log, ddt_bias, dh0 and,
    with the norm, dO, dg, dw."""
    if not ctx.saved:
        raise ValueError("the forward saved nothing: call kda_forward_conv with save_for_backward=True")
    x = ctx.x
    B, T, _ = x.shape
    H, dk, dv = ctx.A_log.shape[0], ctx.dk, ctx.dv
    _shape(dy, "dy", (B, T, H, dv))
    _check(dy, "dy", x.dtype)
    if dh_final is not None:
        _shape(dh_final, "dh_final", (ctx.n_docs, H, dk, dv))
        _check(dh_final, "dh_final", torch.float32)
    norm = ctx.g is not None
    gr = {
        "dx": torch.empty_like(x), "dconv_w": torch.empty_like(ctx.conv_w), "df": torch.empty_like(ctx.f),
        "db": torch.empty_like(ctx.b), "dA_log": torch.empty(H, dtype=torch.float32, device=x.device),
        "ddt_bias": torch.empty_like(ctx.dt_bias),
        "dh0": torch.empty(ctx.n_docs, H, dk, dv, dtype=torch.float32, device=x.device) if want_dh0 else None,
        "dO": torch.empty_like(dy) if norm else None, "dg": torch.empty_like(dy) if norm else None,
        "dw": torch.empty(dv, dtype=torch.float32, device=x.device) if norm else None,
    }
    _lib.kda_bwd_conv(ctx.problem, x, ctx.conv_w, ctx.f, ctx.b, ctx.A_log, ctx.dt_bias, ctx.h0, ctx.g, ctx.w, ctx.eps,
                      dy, dh_final, gr["dO"], gr["dg"], gr["dw"], gr["dx"], gr["dconv_w"], gr["df"], gr["db"],
                      gr["dA_log"], gr["ddt_bias"], gr["dh0"], ctx.workspace)
    return gr


def kda_decode_step(q, k, v, f, b, A_log, dt_bias, state, scale: Optional[float] = None,
                    out: Optional[torch.Tensor] = None):
    """One token for each of n sequences: q, k, f [n, H, dk] (or f [n, H] for
    the scalar gate), v [n, H, dv], b [n, H] (bf16 or fp32), state
    [n, H, dk, dv] fp32 updated in place.
    Returns o [n, H, dv] in the io dtype."""
    _dims(q, "q", 3)
    _dims(v, "v", 3)
    n, H, dk = q.shape
    dv = v.shape[-1]
    _shape(k, "k", q.shape)
    _shape(b, "b", (n, H))
    _shape(A_log, "A_log", (H,))
    _shape(state, "state", (n, H, dk, dv))
    gate = _gate_of(f, dt_bias, (n, H, dk))
    if out is not None:
        _shape(out, "out", (n, H, dv))
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (f, "f"), (b, "b")):
        _check(t, nm, q.dtype)
    _check(A_log, "A_log", torch.float32)
    _check(dt_bias, "dt_bias", torch.float32)
    _check(state, "state", torch.float32)
    if out is not None:
        _check(out, "out", q.dtype)
    o = out if out is not None else torch.empty(n, H, dv, dtype=q.dtype, device=q.device)
    _lib.kda_decode(n, H, dk, dv, q.dtype, scale, q, k, v, f, b, A_log, dt_bias, state, o, gate)
    return o


def _norm_args(x, g, w):
    _shape(g, "g", x.shape)
    _shape(w, "w", (x.shape[-1],))
    _check(x, "x")
    _check(g, "g", x.dtype)
    _check(w, "w", torch.float32)


def _conv_args(x, w, cu_seqlens):
    _shape(w, "w", (x.shape[-1], 4))
    if cu_seqlens is not None:
        _dims(cu_seqlens, "cu_seqlens", 1)
    _check(x, "x")
    _check(w, "w", torch.float32)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32)


def kda_norm_gate(x, g, w, eps: Optional[float] = None, out: Optional[torch.Tensor] = None):
    """Gated RMSNorm epilogue over the last axis (dv = 64 or 128):
    y = x / sqrt(mean(x^2) + eps) * w * sigmoid(g); x, g [..., dv] (bf16 or
    fp32, e.g. the KDA output [B, T, H, dv]), w [dv] fp32."""
    _norm_args(x, g, w)
    if out is not None:
        _shape(out, "out", x.shape)
        _check(out, "out", x.dtype)
    dv = x.shape[-1]
    y = out if out is not None else torch.empty_like(x)
    _lib.kda_norm_gate_fwd(x.numel() // dv, dv, x.dtype, eps, x, g, w, y)
    return y


def kda_norm_gate_backward(x, g, w, dy, eps: Optional[float] = None, workspace: Optional[torch.Tensor] = None):
    """Backward of kda_norm_gate: returns (dx, dg, dw)."""
    _shape(dy, "dy", x.shape)
    _norm_args(x, g, w)
    _check(dy, "dy", x.dtype)
    dv = x.shape[-1]
    n = x.numel() // dv
    if workspace is None:
        workspace = torch.empty(_lib.kda_norm_gate_workspace_size(n, dv), dtype=torch.uint8, device=x.device)
    dx, dg = torch.empty_like(x), torch.empty_like(g)
    dw = torch.empty_like(w)
    _lib.kda_norm_gate_bwd(n, dv, x.dtype, eps, x, g, w, dy, dx, dg, dw, workspace)
    return dx, dg, dw


def kda_short_conv(x, w, cu_seqlens=None, activation: str = "silu", out: Optional[torch.Tensor] = None):
    """Short causal depthwise convolution (width 4) over tokens, reset at the
    cu_seqlens document starts: x [..., C] token-major (e.g. the concatenated
    q | k | v projections [B, T, C]), w [C, 4] fp32; activation "silu" or
    "none"."""
    _conv_args(x, w, cu_seqlens)
    if out is not None:
        _shape(out, "out", x.shape)
        _check(out, "out", x.dtype)
    C = x.shape[-1]
    y = out if out is not None else torch.empty_like(x)
    _lib.kda_short_conv_fwd(x.numel() // C, C, x.dtype, 1 if activation == "silu" else 0, cu_seqlens, x, w, y)
    return y


def kda_short_conv_backward(x, w, dy, cu_seqlens=None, activation: str = "silu",
                            workspace: Optional[torch.Tensor] = None):
    """Backward of kda_short_conv: returns (dx, dw)."""
    _shape(dy, "dy", x.shape)
    _conv_args(x, w, cu_seqlens)
    _check(dy, "dy", x.dtype)
    C = x.shape[-1]
    n = x.numel() // C
    if workspace is None:
        workspace = torch.empty(_lib.kda_short_conv_workspace_size(n, C), dtype=torch.uint8, device=x.device)
    dx, dw = torch.empty_like(x), torch.empty_like(w)
    _lib.kda_short_conv_bwd(n, C, x.dtype, 1 if activation == "silu" else 0, cu_seqlens, x, w, dy, dx, dw, workspace)
    return dx, dw


from .autograd import gated_norm, kda_attention, short_conv  # noqa: E402  (differentiable forms)
