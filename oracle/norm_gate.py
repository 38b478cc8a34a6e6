"""Plain CPU oracle of the gated RMSNorm output epilogue (float64 numpy).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg
use it; the CUDA library never does.

Operation, per token and head over the value dimension dv ("Pure KDA 300M"
guide, Overview: per-head output gate and RMSNorm with eps = 1e-6; the
openkimi README, "What is implemented": FLA's fused RMSNorm plus sigmoid
gate on the KDA output):
    r   = 1 / sqrt(mean_j x_j^2 + eps)
    y_j = x_j * r * w_j * sigmoid(g_j)
with one weight vector w [dv] shared by the heads (a reading: the pages name
a per-head norm of width head_v_dim, whose weight has dv entries).

Backward of L with dy = dL/dy, written out by the chain rule:
    s_j  = sigmoid(g_j),  xh_j = x_j r
    dg_j = dy_j xh_j w_j s_j (1 - s_j)
    dw_j = sum over rows of dy_j xh_j s_j
    a_j  = dy_j w_j s_j                      (dL/dxh_j)
    dx_j = r (a_j - xh_j mean_k(a_k xh_k))   (the RMSNorm Jacobian)
Rows are the leading axes flattened: x, g, dy [N, dv]; w [dv].
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def forward(x, g, w, eps: float = EPS):
    x = np.asarray(x, np.float64)
    g = np.asarray(g, np.float64)
    w = np.asarray(w, np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * w * _sigmoid(g)


def backward(x, g, w, dy, eps: float = EPS):
    """Returns (dx, dg, dw)."""
    x = np.asarray(x, np.float64)
    g = np.asarray(g, np.float64)
    w = np.asarray(w, np.float64)
    dy = np.asarray(dy, np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    s = _sigmoid(g)
    xh = x * r
    dg = dy * xh * w * s * (1.0 - s)
    dw = (dy * xh * s).reshape(-1, x.shape[-1]).sum(axis=0)
    a = dy * w * s
    dx = r * (a - xh * np.mean(a * xh, axis=-1, keepdims=True))
    return dx, dg, dw
