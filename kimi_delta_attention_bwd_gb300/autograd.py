"""torch.autograd integration of the KDA operations: the same library calls
as kda_forward / kda_backward (and the convolution and gated-norm entry
points), wrapped so that a model can use them like any differentiable op.

  o = kda_attention(q, k, v, f, b, A_log, dt_bias)                    # o
  o, h_final = kda_attention(..., h0=h0, output_final_state=True)     # and the final states
  x = short_conv(x_raw, conv_w, cu_seqlens)                           # causal conv (k=4) + silu
  y = gated_norm(o, gate, weight)                                     # gated RMSNorm epilogue

Gradients flow to q, k, v, f, b, A_log, dt_bias and h0 (and to the
convolution's input and taps, the norm's input, gate and weight).  Each
backward runs the library's backward kernels once; a second derivative is
not provided.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import kda_backward, kda_forward, kda_norm_gate, kda_norm_gate_backward, kda_short_conv, kda_short_conv_backward

__all__ = ["kda_attention", "short_conv", "gated_norm"]


class _KdaAttention(torch.autograd.Function):
    @staticmethod
    def forward(fctx, q, k, v, f, b, A_log, dt_bias, h0, scale, cu_seqlens, cu_seqlens_host, want_final):
        o, hf, kctx = kda_forward(q, k, v, f, b, A_log, dt_bias, scale=scale, h0=h0, cu_seqlens=cu_seqlens,
                                  cu_seqlens_host=cu_seqlens_host, save_for_backward=True,
                                  want_final_state=want_final)
        fctx.kctx = kctx
        fctx.has_h0 = h0 is not None
        if want_final:
            return o, hf
        return o

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(fctx, dO, dhf=None):
        kctx = fctx.kctx
        if dO is None:
            dO = torch.zeros(*kctx.q.shape[:3], kctx.v.shape[-1], dtype=kctx.q.dtype, device=kctx.q.device)
        g = kda_backward(kctx, dO.contiguous(), None if dhf is None else dhf.contiguous(),
                         want_dh0=fctx.has_h0 and fctx.needs_input_grad[7])
        return (g["dq"], g["dk"], g["dv"], g["df"], g["db"], g["dA_log"], g["ddt_bias"],
                g["dh0"] if fctx.has_h0 else None, None, None, None, None)


def kda_attention(q, k, v, f, b, A_log, dt_bias, scale: Optional[float] = None, h0=None, cu_seqlens=None,
                  cu_seqlens_host=None, output_final_state: bool = False):
    """Differentiable KDA: o (and h_final when output_final_state) from the
    layouts of kda_forward; backward through kda_backward."""
    return _KdaAttention.apply(q, k, v, f, b, A_log, dt_bias, h0, scale, cu_seqlens, cu_seqlens_host,
                               output_final_state)


class _ShortConv(torch.autograd.Function):
    @staticmethod
    def forward(fctx, x, w, cu_seqlens, activation):
        fctx.save_for_backward(x, w)
        fctx.cu_seqlens, fctx.activation = cu_seqlens, activation
        return kda_short_conv(x, w, cu_seqlens, activation)

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(fctx, dy):
        x, w = fctx.saved_tensors
        dx, dw = kda_short_conv_backward(x, w, dy.contiguous(), fctx.cu_seqlens, fctx.activation)
        return dx, dw, None, None


def short_conv(x, w, cu_seqlens=None, activation: str = "silu"):
    """Differentiable short causal depthwise convolution (kda_short_conv)."""
    return _ShortConv.apply(x, w, cu_seqlens, activation)


class _GatedNorm(torch.autograd.Function):
    @staticmethod
    def forward(fctx, x, g, w, eps):
        fctx.save_for_backward(x, g, w)
        fctx.eps = eps
        return kda_norm_gate(x, g, w, eps)

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(fctx, dy):
        x, g, w = fctx.saved_tensors
        dx, dg, dw = kda_norm_gate_backward(x, g, w, dy.contiguous(), fctx.eps)
        return dx, dg, dw, None


def gated_norm(x, g, w, eps: Optional[float] = None):
    """Differentiable gated RMSNorm epilogue (kda_norm_gate)."""
    return _GatedNorm.apply(x, g, w, eps)
