"""Failure detection on the GPU without a fault: the bounded waits.

Every mbarrier wait in the library's kernels gives up after a bounded time,
flags KDA_ERR_DEVICE (-7) and returns.  kda_test_stage_timeout(1) makes the
forward state chain's stage barriers expect 16 bytes more than each bulk copy
delivers (the copies themselves all complete), so the waits run out; the test
checks that the call returns, that kda_device_status reports -7 and that the
next, normal call on the same context gives correct results.  Covered: the
plain state chain and the clustered one with the gated norm fused in (whose
two CTAs must both reach their final cluster barrier), each also on a
40-chunk row at two heads, whose chain runs split: there the composing
kernel's waits run out first and the chain kernel then does no steps.
"""
import time

import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import _lib, kda_device_status, kda_forward, kda_forward_norm_gate
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs, norm_gate_inputs
from _common import TOL_IO, rel_max, run_oracle

pytestmark = pytest.mark.gpu


def _run(norm, split):
    T = 64 * 40 if split else 192
    w = custom(1, T, 2, 32, 64, h0=True)
    inp = make_inputs(w, seed=51, with_grad_inputs=False)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    x = (d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"])
    prob = _lib.make_problem(1, T, 2, 32, 64, torch.bfloat16, d["scale"])
    ws = _lib.alloc_workspace(prob, 0)
    if norm:
        ng = norm_gate_inputs(T * 2, 64, seed=52)
        g, wn = ng["g"].reshape(1, T, 2, 64).cuda(), ng["w"].cuda()
        y, _, _, _ = kda_forward_norm_gate(*x, g, wn, scale=d["scale"], h0=d["h0"], save_for_backward=False,
                                           workspace=ws)
        return y, ws, inp
    o, _, _ = kda_forward(*x, scale=d["scale"], h0=d["h0"], save_for_backward=False, workspace=ws)
    return o, ws, inp


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("norm", [False, True])
def test_stage_wait_runs_out_and_context_survives(norm, split):
    lib = _lib.load()
    if split:  # the row does run split
        _lib.prof_start()
        _run(norm, split)
        torch.cuda.synchronize()
        assert _lib.prof_stop()["fwd_seg"][1] == 1
    lib.kda_test_stage_timeout(1)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        _, ws, _ = _run(norm, split)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert kda_device_status(ws) == -7
    finally:
        lib.kda_test_stage_timeout(0)
    print(f"\n[wait run-out] norm={norm} split={split}: the forward returned after {elapsed:.2f} s")
    assert elapsed < 60.0
    out, ws, inp = _run(norm, split)  # the same context, normal waits
    assert kda_device_status(ws) == 0
    T = out.shape[1]
    if not norm:
        ref = run_oracle(inp, False)
        assert rel_max(out.double().cpu().numpy().reshape(T, 2, 64), ref["o"], bf16=True) <= TOL_IO
    assert np.isfinite(out.float().cpu().numpy()).all()
