"""Plain CPU oracle of the varlen short causal depthwise convolution that
precedes the KDA path (float64 numpy).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg
use it; the CUDA library never does.

Operation ("Pure KDA 300M" guide, Overview: short-conv kernel size 4,
depthwise, on the concatenated QKV; the guide's troubleshooting section uses
FLA's causal_conv1d, which takes [B, T, D] directly; torchtitan's sample
packing resets per document at cu_seqlens):
    z_t,c = sum_{j=0}^{K-1} w_c,j x_{t-K+1+j, c}     (x before the document start is 0)
    y_t,c = silu(z_t,c) = z sigmoid(z)                 (activation "silu"; "none": y = z)
over tokens t of each document and channels c, x [Ntok, C], w [C, K].

Backward, from the definition: dz = dy silu'(z) with silu'(z) = s (1 + z (1 - s)),
s = sigmoid(z); dx_t = sum_j w_j dz_{t+K-1-j} (same document); dw_c,j = sum_t
dz_t,c x_{t-K+1+j, c}.
"""
from __future__ import annotations

import numpy as np


def _docs(n, cu):
    if cu is None:
        return [(0, n)]
    cu = [int(v) for v in cu]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def _pre(x, w, a, b):
    """z for the tokens [a, b) of one document."""
    K = w.shape[1]
    z = np.zeros((b - a, x.shape[1]))
    for j in range(K):
        shift = K - 1 - j  # z_t uses x_{t - shift}
        if shift < b - a:
            z[shift:] += w[:, j] * x[a:b - shift]
    return z


def forward(x, w, cu=None, activation: str = "silu"):
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    y = np.zeros_like(x)
    for a, b in _docs(x.shape[0], cu):
        if b > a:
            z = _pre(x, w, a, b)
            y[a:b] = z / (1.0 + np.exp(-z)) if activation == "silu" else z
    return y


def backward(x, w, dy, cu=None, activation: str = "silu"):
    """Returns (dx, dw)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    dy = np.asarray(dy, np.float64)
    K = w.shape[1]
    dx = np.zeros_like(x)
    dw = np.zeros_like(w)
    for a, b in _docs(x.shape[0], cu):
        if b <= a:
            continue
        z = _pre(x, w, a, b)
        if activation == "silu":
            s = 1.0 / (1.0 + np.exp(-z))
            dz = dy[a:b] * s * (1.0 + z * (1.0 - s))
        else:
            dz = dy[a:b]
        for j in range(K):
            shift = K - 1 - j
            if shift < b - a:
                dx[a:b - shift] += w[:, j] * dz[shift:]
                dw[:, j] += (dz[shift:] * x[a:b - shift]).sum(axis=0)
    return dx, dw
