"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/kda.h declares, sizes its workspace, and rejects
bad arguments on the host before any launch.  Every call below is built to
fail validation, so no kernel is ever launched with the fake pointers."""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import _lib

FAKE = 1 << 20  # 256-byte aligned non-null fake address; never dereferenced


def test_exports_every_declared_symbol():
    lib = _lib.load()
    names = _lib.exported_names()
    assert {"kda_fwd", "kda_bwd", "kda_workspace_size", "kda_strerror", "kda_device_status",
            "kda_prof_start", "kda_prof_stop", "kda_prof_kernel_name"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_and_kernel_names():
    lib = _lib.load()
    for s in range(-7, 1):
        assert len(lib.kda_strerror(s)) > 0
    names = []
    i = 0
    while lib.kda_prof_kernel_name(i) is not None:
        names.append(lib.kda_prof_kernel_name(i).decode())
        i += 1
    assert "bwd_intra" in names and "fwd_scan" in names


def prob(**kw):
    a = dict(B=2, T=100, H=4, dk=32, dv=64, dtype=torch.bfloat16)
    a.update(kw)
    cu = a.pop("cu", None)
    cu_host = a.pop("cu_host", None)
    p = _lib.make_problem(a["B"], a["T"], a["H"], a["dk"], a["dv"], a["dtype"])
    if cu is not None:
        p.cu_seqlens = cu
        p.n_docs = a.get("n_docs", 2)
    if cu_host is not None:
        p.cu_seqlens_host = cu_host.ctypes.data
    return p


def test_workspace_size_rules():
    lib = _lib.load()
    p = prob()
    f = lib.kda_workspace_size(ctypes.byref(p), 0)
    b = lib.kda_workspace_size(ctypes.byref(p), 1)
    assert 0 < f < b and f % 256 == 0 and b % 256 == 0
    assert lib.kda_workspace_size(ctypes.byref(prob(dk=48)), 0) == 0      # unsupported
    assert lib.kda_workspace_size(ctypes.byref(prob(T=0)), 0) == 0        # invalid
    assert lib.kda_workspace_size(None, 0) == 0
    big = lib.kda_workspace_size(ctypes.byref(prob(T=1000)), 1)
    assert big > b


def call_fwd(p, ptr=FAKE, ws=FAKE, ws_bytes=1 << 40, o=FAKE):
    lib = _lib.load()
    P = ctypes.c_void_p
    return lib.kda_fwd(ctypes.byref(p), P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), None,
                       P(o), None, 1, P(ws), ws_bytes, None)


def call_bwd(p, ptr=FAKE, ws=FAKE, ws_bytes=1 << 40):
    lib = _lib.load()
    P = ctypes.c_void_p
    args = [P(ptr)] * 7 + [None, P(ptr), None] + [P(ptr)] * 7 + [None]
    return lib.kda_bwd(ctypes.byref(p), *args, P(ws), ws_bytes, None)


def test_host_validation_statuses():
    assert call_fwd(prob(dk=48)) == -2                   # unsupported head shape
    assert call_fwd(prob(dtype=torch.float16)) == -1     # unsupported dtype
    assert call_fwd(prob(H=0)) == -1
    assert call_fwd(prob(), ptr=0) == -1                 # null input
    assert call_fwd(prob(), o=0) == -1                   # null output
    assert call_fwd(prob(), ptr=FAKE + 2) == -3          # misaligned input
    assert call_fwd(prob(), ws=FAKE + 16) == -3          # workspace not 256-aligned
    assert call_fwd(prob(), ws=0) == -5
    assert call_fwd(prob(), ws_bytes=1024) == -5         # workspace too small
    assert call_bwd(prob(dk=100)) == -2
    assert call_bwd(prob(), ptr=0) == -1
    assert call_bwd(prob(), ws_bytes=16) == -5


def test_host_copy_of_offsets_is_validated():
    good = np.array([0, 120, 200], dtype=np.int32)
    for bad in ([0, 120, 199], [1, 120, 200], [0, 150, 120]):
        cu = np.array(bad, dtype=np.int32)
        assert call_fwd(prob(cu=FAKE, cu_host=cu, n_docs=2)) == -4
    # a good host copy passes validation and then stops at the small workspace
    assert call_fwd(prob(cu=FAKE, cu_host=good, n_docs=2), ws_bytes=64) == -5
    # a host copy without the device array is an argument error
    p = prob()
    p.cu_seqlens_host = good.ctypes.data
    assert call_fwd(p) == -1
    # a zero-document list is an argument error
    assert call_fwd(prob(cu=FAKE, cu_host=good, n_docs=0)) == -1


def test_binding_refuses_non_cuda_tensors():
    from kimi_delta_attention_bwd_gb300 import kda_forward
    x = torch.zeros(1, 4, 1, 32)
    with pytest.raises(ValueError):
        kda_forward(x, x, torch.zeros(1, 4, 1, 64), x, torch.zeros(1, 4, 1), torch.zeros(1), torch.zeros(1, 32),
                    scale=None)


def _fwd_args(B=1, T=4, H=2, dk=32, dv=64):
    return dict(q=torch.zeros(B, T, H, dk), k=torch.zeros(B, T, H, dk), v=torch.zeros(B, T, H, dv),
                f=torch.zeros(B, T, H, dk), b=torch.zeros(B, T, H), A_log=torch.zeros(H), dt_bias=torch.zeros(H, dk))


@pytest.mark.parametrize("name,bad", [("k", (1, 4, 2, 16)), ("v", (1, 3, 2, 64)), ("b", (1, 4, 1)),
                                      ("A_log", (3,)), ("dt_bias", (2, 16)), ("f", (1, 4, 2, 8)),
                                      ("h0", (2, 2, 32, 64)), ("out", (1, 4, 2, 32))])
def test_binding_rejects_mismatched_shapes_before_any_launch(name, bad):
    # the C ABI sees pointers only: a tensor smaller than its layout would be read out of bounds, so the
    # binding checks every shape first (these CPU tensors never reach the library)
    from kimi_delta_attention_bwd_gb300 import kda_forward
    a = _fwd_args()
    a[name] = torch.zeros(bad)
    with pytest.raises(ValueError, match=name):
        kda_forward(**a)


def test_backward_and_epilogue_bindings_reject_mismatched_shapes():
    from kimi_delta_attention_bwd_gb300 import (KdaContext, kda_backward, kda_decode_step, kda_norm_gate,
                                                kda_norm_gate_backward, kda_short_conv, kda_short_conv_backward)
    a = _fwd_args()
    ctx = KdaContext(None, a["q"], a["k"], a["v"], a["f"], a["b"], a["A_log"], a["dt_bias"], None, None, None, None, 1)
    with pytest.raises(ValueError, match="dO"):
        kda_backward(ctx, torch.zeros(1, 4, 2, 32))
    with pytest.raises(ValueError, match="dh_final"):
        kda_backward(ctx, torch.zeros(1, 4, 2, 64), torch.zeros(2, 2, 32, 64))
    with pytest.raises(ValueError, match="dq"):
        kda_backward(ctx, torch.zeros(1, 4, 2, 64), grads={"dq": torch.zeros(1, 4, 2, 16)})
    d = {n: t[0] for n, t in a.items() if n not in ("A_log", "dt_bias")}  # one token of 4 sequences
    with pytest.raises(ValueError, match="b"):
        kda_decode_step(d["q"], d["k"], d["v"], d["f"], torch.zeros(4, 3), a["A_log"], a["dt_bias"],
                        torch.zeros(4, 2, 32, 64))
    with pytest.raises(ValueError, match="state"):
        kda_decode_step(d["q"], d["k"], d["v"], d["f"], d["b"], a["A_log"], a["dt_bias"], torch.zeros(4, 2, 32, 32))
    x = torch.zeros(10, 64)
    with pytest.raises(ValueError, match="g"):
        kda_norm_gate(x, torch.zeros(10, 32), torch.zeros(64))
    with pytest.raises(ValueError, match="w"):
        kda_norm_gate_backward(x, x, torch.zeros(32), x)
    with pytest.raises(ValueError, match="dy"):
        kda_norm_gate_backward(x, x, torch.zeros(64), torch.zeros(9, 64))
    with pytest.raises(ValueError, match="w"):
        kda_short_conv(x, torch.zeros(64, 3))
    with pytest.raises(ValueError, match="dy"):
        kda_short_conv_backward(x, torch.zeros(64, 4), torch.zeros(10, 32))
