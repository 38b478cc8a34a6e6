"""Python front end of the plain CPU KDA oracle (kda_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg call this; the CUDA library never does.

The C code runs one (document, head) unit at a time, token by token.  Units
are independent, so this wrapper spreads disjoint unit lists over Python
threads (ctypes releases the GIL during the call); each thread writes only
the rows and states of its own units, and the per-unit parameter-gradient
partials are summed here in float64.

Arrays use the flattened token-major layout:
  q, k, f [Ntok, H, dk]; v, o, dO [Ntok, H, dv]; b [Ntok, H];
  A_log [H]; dt_bias [H, dk]; states [n_seqs, H, dk, dv].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.c")
BUILD = os.path.join(HERE, "_build")
EPS = 1e-6  # L2-norm epsilon (a reading: the pages give none)

_libs: dict = {}
_lock = threading.Lock()


def lib_path(precision: str = "f64") -> str:
    return os.path.join(BUILD, f"libkda_oracle_{precision}.so")


def build(precision: str = "f64", force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    out = lib_path(precision)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(BUILD, exist_ok=True)
    real = {"f64": "double", "f32": "float"}[precision]
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           f"-DORACLE_REAL={real}", "-o", tmp, SRC, "-lm"])
    os.replace(tmp, out)
    return out


def declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Sets the argument and return types of the oracle's C entry points."""
    P = ctypes.c_void_p
    i, d = ctypes.c_int, ctypes.c_double
    lib.kda_oracle_forward.argtypes = [i, i, i, i, P, P, P, P, P, P, P, d, d, i, P, P, i, P, P, P, P]
    lib.kda_oracle_forward.restype = i
    lib.kda_oracle_backward.argtypes = [i, i, i, i, P, P, P, P, P, P, P, d, d, i, P, P, P, P,
                                        i, P, P, P, P, P, P, P, P, P]
    lib.kda_oracle_backward.restype = i
    lib.kda_oracle_gate.argtypes = [d, d]
    lib.kda_oracle_gate.restype = d
    lib.kda_oracle_sigmoid.argtypes = [d]
    lib.kda_oracle_sigmoid.restype = d
    lib.kda_oracle_real_bytes.restype = i
    return lib


def load(precision: str = "f64") -> ctypes.CDLL:
    with _lock:
        if precision in _libs:
            return _libs[precision]
        lib = declare(ctypes.CDLL(build(precision)))
        _libs[precision] = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _units(cu, H, units):
    if units is None:
        n = len(cu) - 1
        units = [(s, h) for s in range(n) for h in range(H)]
    us = np.ascontiguousarray([u[0] for u in units], dtype=np.int32)
    uh = np.ascontiguousarray([u[1] for u in units], dtype=np.int32)
    return us, uh


def _split(n, parts, cu=None, us=None):
    """Split range(n) into contiguous pieces of similar token work."""
    parts = max(1, min(parts, n))
    if cu is None or us is None:
        bounds = np.linspace(0, n, parts + 1).astype(int)
        return [(bounds[i], bounds[i + 1]) for i in range(parts)]
    w = (cu[us + 1] - cu[us]).astype(np.float64) + 1.0
    cw = np.concatenate([[0.0], np.cumsum(w)])
    tgt = np.linspace(0, cw[-1], parts + 1)
    idx = np.searchsorted(cw, tgt[1:-1])
    cuts = [0] + sorted(set(int(x) for x in idx)) + [n]
    return [(cuts[i], cuts[i + 1]) for i in range(len(cuts) - 1) if cuts[i + 1] > cuts[i]]


def default_threads():
    return max(1, os.cpu_count() or 1)


def forward(x: dict, units=None, threads: int | None = None, precision: str = "f64"):
    """Run the forward recurrence.  x holds float64 arrays q, k, v, f, b,
    A_log, dt_bias, optional h0, int32 cu_seqlens and float scale.  Returns
    (o, h_final); rows/states of units not listed are left at zero."""
    lib = load(precision)
    q, k, v, f, b = (_c64(x[n]) for n in ("q", "k", "v", "f", "b"))
    A_log, dtb, h0 = _c64(x["A_log"]), _c64(x["dt_bias"]), _c64(x.get("h0"))
    cu = np.ascontiguousarray(x["cu_seqlens"], dtype=np.int32)
    Ntok, H, dk = q.shape
    dv = v.shape[2]
    n_seqs = len(cu) - 1
    us, uh = _units(cu, H, units)
    o = np.zeros((Ntok, H, dv))
    hf = np.zeros((n_seqs, H, dk, dv))
    eps = float(x.get("eps", EPS))

    def run(lo, hi):
        if hi <= lo:
            return 0
        return lib.kda_oracle_forward(Ntok, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(b),
                                      _ptr(A_log), _ptr(dtb), float(x["scale"]), eps,
                                      n_seqs, _ptr(cu), _ptr(h0), hi - lo,
                                      _ptr(us[lo:]), _ptr(uh[lo:]), _ptr(o), _ptr(hf))
    pieces = _split(len(us), threads or default_threads(), cu, us)
    with ThreadPoolExecutor(len(pieces)) as ex:
        rcs = list(ex.map(lambda p: run(*p), pieces))
    if any(rcs):
        raise ValueError("oracle forward rejected its arguments")
    return o, hf


def backward(x: dict, dO, dh_final=None, units=None, threads: int | None = None, precision: str = "f64"):
    """Reverse-mode gradients of  sum(o*dO) + sum(h_final*dh_final).
    Returns a dict dq, dk, dv, df, db, dA_log, ddt_bias, dh0 (float64)."""
    lib = load(precision)
    q, k, v, f, b = (_c64(x[n]) for n in ("q", "k", "v", "f", "b"))
    A_log, dtb, h0 = _c64(x["A_log"]), _c64(x["dt_bias"]), _c64(x.get("h0"))
    dO, dhf = _c64(dO), _c64(dh_final)
    cu = np.ascontiguousarray(x["cu_seqlens"], dtype=np.int32)
    Ntok, H, dk = q.shape
    dv = v.shape[2]
    n_seqs = len(cu) - 1
    us, uh = _units(cu, H, units)
    n = len(us)
    g = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
         "df": np.zeros_like(f), "db": np.zeros_like(b), "dh0": np.zeros((n_seqs, H, dk, dv))}
    dAp = np.zeros(n)
    ddp = np.zeros((n, dk))
    eps = float(x.get("eps", EPS))

    def run(lo, hi):
        if hi <= lo:
            return 0
        return lib.kda_oracle_backward(Ntok, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(f), _ptr(b),
                                       _ptr(A_log), _ptr(dtb), float(x["scale"]), eps,
                                       n_seqs, _ptr(cu), _ptr(h0), _ptr(dO), _ptr(dhf), hi - lo,
                                       _ptr(us[lo:]), _ptr(uh[lo:]),
                                       _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["df"]), _ptr(g["db"]),
                                       _ptr(dAp[lo:]), _ptr(ddp[lo:]), _ptr(g["dh0"]))
    pieces = _split(n, threads or default_threads(), cu, us)
    with ThreadPoolExecutor(len(pieces)) as ex:
        rcs = list(ex.map(lambda p: run(*p), pieces))
    if any(rcs):
        raise ValueError("oracle backward rejected its arguments")
    dA = np.zeros(H)
    dd = np.zeros((H, dk))
    for i in range(n):  # fixed order: deterministic sums
        dA[uh[i]] += dAp[i]
        dd[uh[i]] += ddp[i]
    g["dA_log"] = dA
    g["ddt_bias"] = dd
    return g


def gate(A_log: float, x: float, precision: str = "f64") -> float:
    return load(precision).kda_oracle_gate(float(A_log), float(x))


def sigmoid(x: float, precision: str = "f64") -> float:
    return load(precision).kda_oracle_sigmoid(float(x))
