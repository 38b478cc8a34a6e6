"""Seeded synthetic inputs for the KDA workloads.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic.  The oracle and the CUDA path both take their inputs
from here, so that they see bit-identical values (the oracle receives the
io-dtype values widened to float64).

Shapes follow the "Pure KDA 300M" guide (Primus, ROCm docs), Overview:
8 heads, head_k_dim 32, head_v_dim 64, sequence length 2048; one KDA call in
that model sees a micro-batch of 16 rows.  The pages train on FineWeb-Edu,
which is not used here: these seeded draws stand in for it.

Distributions (same for every workload):
  q, k, v, f, b, dO ~ N(0, 1)            (q, k raw; the kernels L2-normalise)
  A_log  = log U[1, 16]                  per head
  dt     ~ log-uniform [1e-3, 1e-1]      per (head, key channel)
  dt_bias = dt + log(-expm1(-dt))        so that softplus(dt_bias) = dt
  h0     ~ N(0, 0.02^2)                  per document and head, when used
  dh_final ~ N(0, 1)                     when used
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

BASE_SEED = 20261202


@dataclass(frozen=True)
class KdaWorkload:
    index: int
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    dtype: str            # "f32" or "bf16": the io dtype of q, k, v, f, b, o, dO and gradients
    backward: bool
    varlen: Optional[str]  # None, "docs600" or "rows8192_docs2048"
    h0: bool
    dh_final: bool
    gate: str = "channel"  # "channel": f [B,T,H,dk], dt_bias [H,dk] (KDA); "scalar": f [B,T,H], dt_bias [H] (GDN)

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = [
    KdaWorkload(0, "tiny fwd+bwd, 1x256, H2, 32/64, fp32", 1, 256, 2, 32, 64, "f32", True, None, False, False),
    KdaWorkload(1, "300M layer fwd, 16x2048, H8, 32/64, bf16", 16, 2048, 8, 32, 64, "bf16", False, None, False, False),
    KdaWorkload(2, "varlen fwd, 1x32768 packed, H8, 32/64, bf16", 1, 32768, 8, 32, 64, "bf16", False, "docs600", False, False),
    KdaWorkload(3, "300M layer fwd+bwd, 16x2048, H8, 32/64, bf16", 16, 2048, 8, 32, 64, "bf16", True, None, False, False),
    KdaWorkload(4, "large-head varlen fwd+bwd, 4x8192, H16, 128/128, bf16, h0", 4, 8192, 16, 128, 128, "bf16", True,
                "rows8192_docs2048", True, True),
]


def custom(B, T, H, dk, dv, dtype="bf16", h0=False, dh_final=False, name="custom", gate="channel") -> KdaWorkload:
    """An ad-hoc workload (edge cases and small parity cases)."""
    return KdaWorkload(99, name, B, T, H, dk, dv, dtype, True, None, h0, dh_final, gate)


def doc_lengths_docs600(total: int, rng: np.random.RandomState) -> list[int]:
    """Log-normal document lengths, median 600 tokens, sigma 1.0 (a reading),
    clipped to [1, 8192], with at least 5% of documents forced to one token.
    Drawing stops when the next document would not fit; what is left (at
    least one token) is a trailing padding run, kept as one segment."""
    lens: list[int] = []
    used = 0
    while True:
        n = int(round(math.exp(rng.normal(math.log(600.0), 1.0))))
        n = min(max(n, 1), 8192)
        if used + n > total - 1:
            break
        lens.append(n)
        used += n
    n_one = max(1, int(math.ceil(0.05 * len(lens))))
    for i in rng.choice(len(lens), size=n_one, replace=False):
        lens[i] = 1
    used = sum(lens)
    lens.append(total - used)  # trailing padding segment
    return lens


def doc_lengths_rows(rows: int, row_len: int, median: float, rng: np.random.RandomState) -> list[int]:
    """Per row, log-normal lengths (sigma 1.0) cut so that documents end at the
    row end; rows are then packed into one flat token axis."""
    lens: list[int] = []
    for _ in range(rows):
        left = row_len
        while left > 0:
            n = int(round(math.exp(rng.normal(math.log(median), 1.0))))
            n = min(max(n, 1), left)
            lens.append(n)
            left -= n
    return lens


def cu_from_lengths(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


def make_inputs(w: KdaWorkload | int, seed: Optional[int] = None, with_grad_inputs: Optional[bool] = None,
                lengths=None):
    """Draw the inputs of one workload.  Returns a dict of CPU tensors:
    q, k, f [B,T,H,dk]; v [B,T,H,dv]; b [B,T,H] in the io dtype;
    A_log [H], dt_bias [H,dk] float32 (scalar gate: f [B,T,H], dt_bias [H]); cu_seqlens int32 [n+1] or None
    (None means equal-length rows; explicit `lengths` override the workload's
    own document draw); h0 [n,H,dk,dv] float32 or None;
    dO [B,T,H,dv] (io dtype) and dh_final float32 or None when the workload
    has a backward; scale (python float)."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    if seed is None:
        seed = BASE_SEED + w.index
    if with_grad_inputs is None:
        with_grad_inputs = w.backward
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.RandomState(seed % (2**32))
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    dt = w.torch_dtype

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dt)

    out = {}
    out["q"] = randn(B, T, H, dk)
    out["k"] = randn(B, T, H, dk)
    out["v"] = randn(B, T, H, dv)
    scalar = w.gate == "scalar"
    out["f"] = randn(B, T, H) if scalar else randn(B, T, H, dk)
    out["b"] = randn(B, T, H)
    u = torch.rand(H, generator=gen, dtype=torch.float64)
    out["A_log"] = torch.log(1.0 + 15.0 * u).to(torch.float32)
    ud = torch.rand(H, generator=gen, dtype=torch.float64) if scalar else torch.rand(H, dk, generator=gen,
                                                                                     dtype=torch.float64)
    dtv = torch.exp(math.log(1e-3) + ud * (math.log(1e-1) - math.log(1e-3)))
    out["dt_bias"] = (dtv + torch.log(-torch.expm1(-dtv))).to(torch.float32)
    if lengths is not None:
        if sum(lengths) != B * T:
            raise ValueError("lengths must sum to B*T")
        cu = cu_from_lengths(lengths)
        n_seqs = len(cu) - 1
    elif w.varlen is None:
        cu = None
        n_seqs = B
    elif w.varlen == "docs600":
        cu = cu_from_lengths(doc_lengths_docs600(B * T, rng))
        n_seqs = len(cu) - 1
    elif w.varlen == "rows8192_docs2048":
        cu = cu_from_lengths(doc_lengths_rows(B, T, 2048.0, rng))
        n_seqs = len(cu) - 1
    else:
        raise ValueError(w.varlen)
    out["cu_seqlens"] = None if cu is None else torch.from_numpy(cu)
    out["h0"] = (0.02 * torch.randn(n_seqs, H, dk, dv, generator=gen, dtype=torch.float32)) if w.h0 else None
    if with_grad_inputs:
        out["dO"] = randn(B, T, H, dv)
        out["dh_final"] = torch.randn(n_seqs, H, dk, dv, generator=gen, dtype=torch.float32) if w.dh_final else None
    out["scale"] = 1.0 / math.sqrt(dk)
    return out


def seq_offsets(inp) -> np.ndarray:
    """Document offsets over the flattened token axis; equal-length rows give
    uniform offsets b*T."""
    if inp.get("cu_seqlens") is not None:
        return inp["cu_seqlens"].numpy().astype(np.int32)
    B, T = inp["q"].shape[0], inp["q"].shape[1]
    return (np.arange(B + 1, dtype=np.int64) * T).astype(np.int32)


def numpy_f64(inp) -> dict:
    """Widen the drawn tensors to float64 numpy arrays in the flattened
    [Ntok, H, d] layout (a lossless conversion of the io-dtype values)."""
    def f64(t):
        return None if t is None else t.to(torch.float64).numpy()
    B, T, H = inp["q"].shape[:3]
    r = {}
    for name in ("q", "k", "v", "f", "dO"):
        if name in inp and inp[name] is not None:
            t = inp[name]
            r[name] = f64(t.reshape(B * T, H, t.shape[-1]) if t.dim() == 4 else t.reshape(B * T, H))
    r["b"] = f64(inp["b"].reshape(B * T, H))
    r["A_log"] = f64(inp["A_log"])
    r["dt_bias"] = f64(inp["dt_bias"])
    r["h0"] = f64(inp.get("h0"))
    r["dh_final"] = f64(inp.get("dh_final"))
    r["cu_seqlens"] = seq_offsets(inp)
    r["scale"] = float(inp["scale"])
    return r


def norm_gate_inputs(n_rows: int, dv: int, dtype: str = "bf16", seed: int = BASE_SEED + 50):
    """Inputs of the gated RMSNorm epilogue: x, g, dy ~ N(0, 1) [n_rows, dv] in
    the io dtype, w ~ 1 + 0.1 N(0, 1) [dv] float32."""
    gen = torch.Generator().manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = torch.randn(n_rows, dv, generator=gen).to(dt)
    g = torch.randn(n_rows, dv, generator=gen).to(dt)
    dy = torch.randn(n_rows, dv, generator=gen).to(dt)
    w = (1.0 + 0.1 * torch.randn(dv, generator=gen)).to(torch.float32)
    return {"x": x, "g": g, "w": w, "dy": dy}


def short_conv_inputs(n_tok: int, C: int, dtype: str = "bf16", seed: int = BASE_SEED + 60):
    """Inputs of the short convolution: x, dy ~ N(0, 1) [n_tok, C] in the io
    dtype, w ~ N(0, 0.5^2) [C, 4] float32."""
    gen = torch.Generator().manual_seed(seed)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = torch.randn(n_tok, C, generator=gen).to(dt)
    dy = torch.randn(n_tok, C, generator=gen).to(dt)
    w = (0.5 * torch.randn(C, 4, generator=gen)).to(torch.float32)
    return {"x": x, "w": w, "dy": dy}
