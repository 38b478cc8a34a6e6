"""Thin ctypes binding of libkda_gb300.so (the C ABI in include/kda.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch provides device memory and the current stream.  There is
no fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

KDA_BF16, KDA_F32 = 0, 1
STATUS = {0: "KDA_OK", -1: "KDA_ERR_INVALID_ARG", -2: "KDA_ERR_UNSUPPORTED", -3: "KDA_ERR_ALIGNMENT",
          -4: "KDA_ERR_BAD_SEQLENS", -5: "KDA_ERR_WORKSPACE", -6: "KDA_ERR_CUDA", -7: "KDA_ERR_DEVICE"}
HEADER = os.path.join(_build.ROOT, "include", "kda.h")


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({strerror(status)})")


class kda_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("n_docs", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("cu_seqlens_host", ctypes.c_void_p), ("gate", ctypes.c_int32)]

KDA_GATE_CHANNEL, KDA_GATE_SCALAR = 0, 1


_lib = None
_lock = threading.Lock()


def exported_names() -> list[str]:
    """Entry points declared in include/kda.h."""
    src = open(HEADER).read()
    return re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", src)


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path) or not _build.up_to_date():
            if not build_if_missing:
                raise RuntimeError(f"CUDA library not built: {path}")
            _build.build()
        lib = ctypes.CDLL(path)
        P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        PP = ctypes.POINTER(kda_problem)
        lib.kda_workspace_size.argtypes = [PP, I]
        lib.kda_workspace_size.restype = SZ
        lib.kda_fwd.argtypes = [PP] + [P] * 10 + [I, P, SZ, P]
        lib.kda_fwd.restype = I
        lib.kda_bwd.argtypes = [PP] + [P] * 18 + [P, SZ, P]
        lib.kda_bwd.restype = I
        lib.kda_device_status.argtypes = [P, P]
        lib.kda_device_status.restype = I
        F = ctypes.c_float
        lib.kda_fwd_norm_gate.argtypes = [PP] + [P] * 10 + [F] + [P] * 3 + [I, P, SZ, P]
        lib.kda_fwd_norm_gate.restype = I
        lib.kda_bwd_norm_gate.argtypes = [PP] + [P] * 10 + [F] + [P] * 13 + [P, SZ, P]
        lib.kda_bwd_norm_gate.restype = I
        lib.kda_fwd_conv.argtypes = [PP] + [P] * 9 + [F] + [P] * 3 + [I, P, SZ, P]
        lib.kda_fwd_conv.restype = I
        lib.kda_bwd_conv.argtypes = [PP] + [P] * 9 + [F] + [P] * 12 + [P, SZ, P]
        lib.kda_bwd_conv.restype = I
        lib.kda_fwd_noalloc.argtypes = [PP] + [P] * 10 + [P]
        lib.kda_fwd_noalloc.restype = I
        lib.kda_test_stage_timeout.argtypes = [I]
        lib.kda_test_stage_timeout.restype = I
        lib.kda_noalloc_status.argtypes = [P]
        lib.kda_noalloc_status.restype = I
        lib.kda_strerror.argtypes = [I]
        lib.kda_strerror.restype = ctypes.c_char_p
        lib.kda_prof_start.restype = I
        lib.kda_prof_stop.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), I]
        lib.kda_prof_stop.restype = I
        lib.kda_prof_kernel_name.argtypes = [I]
        lib.kda_prof_kernel_name.restype = ctypes.c_char_p
        lib.kda_decode.argtypes = [I, I, I, I, I, I, ctypes.c_float] + [P] * 9 + [P]
        lib.kda_decode.restype = I
        I64 = ctypes.c_int64
        lib.kda_norm_gate_workspace_size.argtypes = [I64, I]
        lib.kda_norm_gate_workspace_size.restype = SZ
        lib.kda_norm_gate_fwd.argtypes = [I64, I, I, ctypes.c_float, P, P, P, P, P]
        lib.kda_norm_gate_fwd.restype = I
        lib.kda_norm_gate_bwd.argtypes = [I64, I, I, ctypes.c_float, P, P, P, P, P, P, P, P, SZ, P]
        lib.kda_norm_gate_bwd.restype = I
        lib.kda_short_conv_workspace_size.argtypes = [I64, I]
        lib.kda_short_conv_workspace_size.restype = SZ
        lib.kda_short_conv_fwd.argtypes = [I64, I, I, I, P, I, P, P, P, P]
        lib.kda_short_conv_fwd.restype = I
        lib.kda_short_conv_bwd.argtypes = [I64, I, I, I, P, I, P, P, P, P, P, P, SZ, P]
        lib.kda_short_conv_bwd.restype = I
        _lib = lib
        return lib


def kda_strerror_text(status: int) -> str:
    return strerror(status)


def strerror(status: int) -> str:
    try:
        return load().kda_strerror(int(status)).decode()
    except Exception:  # pragma: no cover
        return "?"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def make_problem(B, T, H, dk, dv, dtype, scale=None, cu_seqlens=None, cu_seqlens_host=None, gate=KDA_GATE_CHANNEL):
    """Builds the kda_problem struct.  cu_seqlens: device int32 tensor or None;
    cu_seqlens_host: host int32 tensor/array kept alive by the caller, or None;
    gate: KDA_GATE_CHANNEL (KDA) or KDA_GATE_SCALAR (scalar-gated GDN)."""
    p = kda_problem()
    p.gate = int(gate)
    p.B, p.T, p.H, p.dk, p.dv = int(B), int(T), int(H), int(dk), int(dv)
    p.dtype = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32 if dtype == torch.float32 else 99
    p.scale = float(scale) if scale is not None else 0.0
    p.n_docs = 0 if cu_seqlens is None else int(cu_seqlens.numel()) - 1
    p.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    p.cu_seqlens_host = None if cu_seqlens_host is None else cu_seqlens_host.ctypes.data if hasattr(
        cu_seqlens_host, "ctypes") else cu_seqlens_host.data_ptr()
    return p


def kda_workspace_size(problem: kda_problem, for_backward) -> int:
    """for_backward: False / 0 (forward only), True / 1 (saving for kda_bwd), 2
    (saving for kda_bwd_norm_gate), 3 (saving for kda_bwd_conv)."""
    kind = int(for_backward) if for_backward in (2, 3) else 1 if for_backward else 0
    return int(load().kda_workspace_size(ctypes.byref(problem), kind))


def alloc_workspace(problem: kda_problem, for_backward, device="cuda") -> torch.Tensor:
    n = kda_workspace_size(problem, for_backward)
    if n == 0:
        raise KdaError(-1, "kda_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)  # torch blocks are 512-byte aligned


def kda_fwd(problem, q, k, v, f, b, A_log, dt_bias, h0, o, h_final, save_for_backward, workspace):
    """Raw forward call; all tensors preallocated on the device."""
    st = load().kda_fwd(ctypes.byref(problem), _p(q), _p(k), _p(v), _p(f), _p(b), _p(A_log), _p(dt_bias),
                        _p(h0), _p(o), _p(h_final), 1 if save_for_backward else 0, _p(workspace),
                        workspace.numel() if workspace is not None else 0, _stream())
    if st != 0:
        raise KdaError(st, "kda_fwd")


def kda_bwd(problem, q, k, v, f, b, A_log, dt_bias, h0, dO, dh_final, dq, dk, dv, df, db,
            dA_log, ddt_bias, dh0, workspace):
    """Raw backward call; all tensors preallocated on the device."""
    st = load().kda_bwd(ctypes.byref(problem), _p(q), _p(k), _p(v), _p(f), _p(b), _p(A_log), _p(dt_bias),
                        _p(h0), _p(dO), _p(dh_final), _p(dq), _p(dk), _p(dv), _p(df), _p(db), _p(dA_log),
                        _p(ddt_bias), _p(dh0), _p(workspace), workspace.numel() if workspace is not None else 0,
                        _stream())
    if st != 0:
        raise KdaError(st, "kda_bwd")


def kda_fwd_norm_gate(problem, q, k, v, f, b, A_log, dt_bias, h0, g, w, eps, o, y, h_final, save_for_backward,
                      workspace):
    """Raw forward with the fused gated RMSNorm epilogue."""
    st = load().kda_fwd_norm_gate(ctypes.byref(problem), _p(q), _p(k), _p(v), _p(f), _p(b), _p(A_log), _p(dt_bias),
                                  _p(h0), _p(g), _p(w), float(eps or 0.0), _p(o), _p(y), _p(h_final),
                                  1 if save_for_backward else 0, _p(workspace),
                                  workspace.numel() if workspace is not None else 0, _stream())
    if st != 0:
        raise KdaError(st, "kda_fwd_norm_gate")


def kda_bwd_norm_gate(problem, q, k, v, f, b, A_log, dt_bias, h0, g, w, eps, dy, dh_final, dO, dg, dw,
                      dq, dk, dv, df, db, dA_log, ddt_bias, dh0, workspace):
    """Raw backward through the fused gated RMSNorm epilogue."""
    st = load().kda_bwd_norm_gate(ctypes.byref(problem), _p(q), _p(k), _p(v), _p(f), _p(b), _p(A_log), _p(dt_bias),
                                  _p(h0), _p(g), _p(w), float(eps or 0.0), _p(dy), _p(dh_final), _p(dO),
                                  _p(dg), _p(dw), _p(dq), _p(dk), _p(dv), _p(df), _p(db), _p(dA_log), _p(ddt_bias),
                                  _p(dh0), _p(workspace), workspace.numel() if workspace is not None else 0,
                                  _stream())
    if st != 0:
        raise KdaError(st, "kda_bwd_norm_gate")


def kda_fwd_conv(problem, x, conv_w, f, b, A_log, dt_bias, h0, g, w, eps, o, y, h_final, save_for_backward,
                 workspace):
    """Raw forward of the layer: short convolution, KDA, optional gated norm."""
    st = load().kda_fwd_conv(ctypes.byref(problem), _p(x), _p(conv_w), _p(f), _p(b), _p(A_log), _p(dt_bias), _p(h0),
                             _p(g), _p(w), float(eps or 0.0), _p(o), _p(y), _p(h_final),
                             1 if save_for_backward else 0, _p(workspace),
                             workspace.numel() if workspace is not None else 0, _stream())
    if st != 0:
        raise KdaError(st, "kda_fwd_conv")


def kda_bwd_conv(problem, x, conv_w, f, b, A_log, dt_bias, h0, g, w, eps, dy, dh_final, dO, dg, dw, dx, dconv_w,
                 df, db, dA_log, ddt_bias, dh0, workspace):
    """Raw backward of the layer."""
    st = load().kda_bwd_conv(ctypes.byref(problem), _p(x), _p(conv_w), _p(f), _p(b), _p(A_log), _p(dt_bias), _p(h0),
                             _p(g), _p(w), float(eps or 0.0), _p(dy), _p(dh_final), _p(dO), _p(dg), _p(dw), _p(dx),
                             _p(dconv_w), _p(df), _p(db), _p(dA_log), _p(ddt_bias), _p(dh0), _p(workspace),
                             workspace.numel() if workspace is not None else 0, _stream())
    if st != 0:
        raise KdaError(st, "kda_bwd_conv")


def kda_decode(n_seq, H, dk, dv, dtype, scale, q, k, v, f, b, A_log, dt_bias, state, o, gate=KDA_GATE_CHANNEL):
    """Raw single-token step; state [n_seq, H, dk, dv] fp32 is updated in place."""
    dt = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32 if dtype == torch.float32 else 99
    st = load().kda_decode(int(n_seq), int(H), int(dk), int(dv), dt, int(gate), float(scale or 0.0), _p(q), _p(k), _p(v),
                           _p(f), _p(b), _p(A_log), _p(dt_bias), _p(state), _p(o), _stream())
    if st != 0:
        raise KdaError(st, "kda_decode")


def _dt(dtype):
    return KDA_BF16 if dtype == torch.bfloat16 else KDA_F32 if dtype == torch.float32 else 99


def kda_norm_gate_fwd(n_rows, dv, dtype, eps, x, g, w, y):
    st = load().kda_norm_gate_fwd(int(n_rows), int(dv), _dt(dtype), float(eps or 0.0), _p(x), _p(g), _p(w), _p(y),
                                  _stream())
    if st != 0:
        raise KdaError(st, "kda_norm_gate_fwd")


def kda_norm_gate_bwd(n_rows, dv, dtype, eps, x, g, w, dy, dx, dg, dw, workspace):
    st = load().kda_norm_gate_bwd(int(n_rows), int(dv), _dt(dtype), float(eps or 0.0), _p(x), _p(g), _p(w), _p(dy),
                                  _p(dx), _p(dg), _p(dw), _p(workspace), workspace.numel(), _stream())
    if st != 0:
        raise KdaError(st, "kda_norm_gate_bwd")


def kda_norm_gate_workspace_size(n_rows, dv) -> int:
    return int(load().kda_norm_gate_workspace_size(int(n_rows), int(dv)))


def kda_short_conv_fwd(n_tok, C, dtype, activation, cu_seqlens, x, w, y):
    nd = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_short_conv_fwd(int(n_tok), int(C), _dt(dtype), int(activation), _p(cu_seqlens), nd, _p(x), _p(w),
                                   _p(y), _stream())
    if st != 0:
        raise KdaError(st, "kda_short_conv_fwd")


def kda_short_conv_bwd(n_tok, C, dtype, activation, cu_seqlens, x, w, dy, dx, dw, workspace):
    nd = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_short_conv_bwd(int(n_tok), int(C), _dt(dtype), int(activation), _p(cu_seqlens), nd, _p(x), _p(w),
                                   _p(dy), _p(dx), _p(dw), _p(workspace), workspace.numel(), _stream())
    if st != 0:
        raise KdaError(st, "kda_short_conv_bwd")


def kda_short_conv_workspace_size(n_tok, C) -> int:
    return int(load().kda_short_conv_workspace_size(int(n_tok), int(C)))


def kda_device_status(workspace) -> int:
    return int(load().kda_device_status(_p(workspace), _stream()))


def prof_start():
    st = load().kda_prof_start()
    if st != 0:
        raise KdaError(st, "kda_prof_start")


def prof_stop() -> dict:
    lib = load()
    names = []
    i = 0
    while True:
        n = lib.kda_prof_kernel_name(i)
        if n is None:
            break
        names.append(n.decode())
        i += 1
    ms = (ctypes.c_double * len(names))()
    cnt = (ctypes.c_int64 * len(names))()
    st = lib.kda_prof_stop(ms, cnt, len(names))
    if st != 0:
        raise KdaError(st, "kda_prof_stop")
    return {names[i]: (ms[i], cnt[i]) for i in range(len(names))}
