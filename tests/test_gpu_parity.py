"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, at every workload's full size, plus the segmentation
identity and the edge cases (partial chunks, one-token and empty documents,
saturated beta, extreme gates, initial states, every compiled head shape).

Tolerances (KDA spec): max|err|/rms(ref) <= 1e-2 for outputs and gradients
(for bf16-stored outputs, after subtracting the half-ulp bf16 rounding of the
exact value, with rms(err)/rms(ref) <= 5e-3 as well), relative Frobenius
error <= 2e-3 for the fp32 final state and dS0; the cu_seqlens segmentation
itself is bit-exact.
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300.inputs import WORKLOADS, custom, make_inputs
from _common import block_spans, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _report(name, errs):
    print(f"\n[parity] {name}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))


@pytest.mark.parametrize("wi", [0, 1, 2, 3])
def test_workload_full_size(wi):
    w = WORKLOADS[wi]
    inp = make_inputs(w)
    gpu = run_gpu(inp, w.backward)
    ref = run_oracle(inp, w.backward)
    _report(w.name, compare(gpu, ref, w.backward, bf16=w.dtype == "bf16"))


def test_varlen_workload_training_step_full_size():
    """The packed varlen row (1 x 32768 tokens, H 8, 32/64, bf16) as a training
    step, with dO: its 128-chunk document makes the batch chain-bound, so both
    state chains run its long documents as composed segments.  Forward and
    backward at full size against the oracle."""
    w = dataclasses.replace(WORKLOADS[2], backward=True)
    inp = make_inputs(w)
    gpu = run_gpu(inp, True)
    ref = run_oracle(inp, True)
    _report(w.name + " (fwd+bwd)", compare(gpu, ref, True))


def test_workload4_sampled_heads():
    """H=16, 128/128, varlen with h0 and dS_final at full size; the oracle runs
    every document of three heads (so dA_log and ddt_bias of those heads are
    complete sums)."""
    w = WORKLOADS[4]
    inp = make_inputs(w)
    gpu = run_gpu(inp, True)
    n_docs = inp["cu_seqlens"].numel() - 1
    heads = [0, 7, 15]
    units = [(s, h) for s in range(n_docs) for h in heads]
    ref = run_oracle(inp, True, units=units)
    errs = compare(gpu, ref, True, rows=(slice(None), heads), states=(slice(None), heads), params_heads=heads)
    _report(w.name, errs)


def test_packed_equals_separate_bitwise_torchtitan_fixture():
    with open(os.path.join(GOLDEN, "torchtitan_packing.json")) as fh:
        fx = json.load(fh)
    lens = fx["lengths"]
    w = custom(1, sum(lens), 4, 32, 64)
    inp = make_inputs(w, seed=5, lengths=lens)
    packed = run_gpu(inp, True)
    for s, (t0, t1) in enumerate(zip(fx["cu_seqlens"][:-1], fx["cu_seqlens"][1:])):
        sub = {k: (v[:, t0:t1].contiguous() if k in ("q", "k", "v", "f", "b", "dO") else v) for k, v in inp.items()}
        sub["cu_seqlens"] = None
        one = run_gpu(sub, True)
        for n in ("o", "dq", "dk", "dv", "df", "db"):
            assert np.array_equal(one[n], packed[n][t0:t1]), n
        assert np.array_equal(one["h_final"][0], packed["h_final"][s])
        assert np.array_equal(one["dh0"][0], packed["dh0"][s])
    joined = dict(inp, cu_seqlens=None)
    j = run_gpu(joined, False)
    assert np.array_equal(j["o"][:96], packed["o"][:96])
    assert not np.allclose(j["o"][96:], packed["o"][96:], atol=1e-3)


def test_general_path_packed_equals_separate_bitwise():
    """The general (large-head) kernels on a packed row of seven documents at
    H 16, 128/128: 448 scan CTAs, more than one wave, dispatched longest
    document first.  Every document's outputs and gradients equal its separate
    run bit for bit, with its own h0 and dS_final."""
    lens = [300, 1, 0, 250, 64, 585, 2]
    w = custom(1, sum(lens), 16, 128, 128, dtype="bf16", h0=True, dh_final=True)
    inp = make_inputs(w, seed=18, lengths=lens)
    packed = run_gpu(inp, True)
    cu = inp["cu_seqlens"].numpy()
    for s in range(len(lens)):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        if t1 == t0:
            assert np.array_equal(packed["h_final"][s], inp["h0"][s].double().numpy()), s
            assert np.array_equal(packed["dh0"][s], inp["dh_final"][s].double().numpy()), s
            continue
        sub = {k: (v[:, t0:t1].contiguous() if k in ("q", "k", "v", "f", "b", "dO") else v) for k, v in inp.items()}
        sub["cu_seqlens"] = None
        sub["h0"] = inp["h0"][s:s + 1].contiguous()
        sub["dh_final"] = inp["dh_final"][s:s + 1].contiguous()
        one = run_gpu(sub, True)
        for n in ("o", "dq", "dk", "dv", "df", "db"):
            assert np.array_equal(one[n], packed[n][t0:t1]), (s, n)
        assert np.array_equal(one["h_final"][0], packed["h_final"][s]), s
        assert np.array_equal(one["dh0"][0], packed["dh0"][s]), s


def test_varlen_workload_segmentation_bitwise():
    """Every document of the packed varlen workload equals its separate run,
    forward and backward (the long documents run as composed segments in both:
    the packed row is chain-bound, and so is a lone document over 32 chunks)."""
    w = dataclasses.replace(WORKLOADS[2], backward=True)
    inp = make_inputs(w)
    packed = run_gpu(inp, True)
    cu = inp["cu_seqlens"].numpy()
    for s in range(len(cu) - 1):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        if t1 == t0:
            continue
        sub = {k: (v[:, t0:t1].contiguous() if k in ("q", "k", "v", "f", "b", "dO") else v) for k, v in inp.items()}
        sub["cu_seqlens"] = None
        one = run_gpu(sub, True)
        for n in ("o", "dq", "dk", "dv", "df", "db"):
            assert np.array_equal(one[n], packed[n][t0:t1]), (s, n)
        assert np.array_equal(one["h_final"][0], packed["h_final"][s]), s


EDGE = {
    "T1": dict(B=2, T=1, H=2, lens=None),
    "ragged_rows": dict(B=3, T=100, H=3, lens=None),
    "one_token_and_empty_docs": dict(B=1, T=200, H=2, lens=[1, 0, 64, 1, 65, 0, 69]),
    "many_tiny_docs": dict(B=1, T=130, H=2, lens=[1] * 70 + [60]),
}


@pytest.mark.parametrize("name", list(EDGE))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_shapes(name, dtype):
    e = EDGE[name]
    w = custom(e["B"], e["T"], e["H"], 32, 64, dtype=dtype, h0=True, dh_final=True)
    inp = make_inputs(w, seed=11, lengths=e["lens"])
    gpu = run_gpu(inp, True)
    ref = run_oracle(inp, True)
    _report(f"{name}/{dtype}", compare(gpu, ref, True, bf16=dtype == "bf16"))


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 128)])
def test_head_shapes(dk, dv):
    w = custom(2, 200, 2, dk, dv, dtype="bf16", h0=True, dh_final=True)
    inp = make_inputs(w, seed=12)
    gpu = run_gpu(inp, True)
    ref = run_oracle(inp, True)
    _report(f"{dk}/{dv}", compare(gpu, ref, True))


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 128)])
@pytest.mark.parametrize("mode", ["edge_docs", "fast_decay", "beta1"])
def test_head_shapes_hard_cases(dk, dv, mode):
    """The large-head kernels on packed documents with one-token, empty and
    partial chunks, on per-token log-decays down to about -60 (in-chunk spans
    far past fp32's exp range) and on beta = 1."""
    lens = [1, 0, 64, 1, 65, 0, 69] if mode == "edge_docs" else None
    w = custom(1 if lens else 2, 200, 2, dk, dv, dtype="bf16", h0=True, dh_final=True)
    inp = make_inputs(w, seed=15, lengths=lens)
    if mode == "fast_decay":
        inp["A_log"].fill_(3.0)
        inp["f"].mul_(3.0).add_(1.0)
    elif mode == "beta1":
        inp["b"].fill_(30.0)
    gpu = run_gpu(inp, True)
    for n, v in gpu.items():
        assert np.isfinite(v).all(), n
    ref = run_oracle(inp, True)
    _report(f"{dk}/{dv} {mode}", compare(gpu, ref, True))


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 128)])
def test_head_shapes_fp32_io(dk, dv):
    """fp32 inputs and outputs on the large-head kernels (split-bf16 tensor-core
    products), packed documents with partial chunks."""
    w = custom(1, 230, 2, dk, dv, dtype="f32", h0=True, dh_final=True)
    inp = make_inputs(w, seed=16, lengths=[100, 1, 129])
    gpu = run_gpu(inp, True)
    ref = run_oracle(inp, True)
    _report(f"{dk}/{dv} f32", compare(gpu, ref, True, bf16=False))


def degenerate(inp, mode):
    """Sets the gate inputs of a drawn problem to one of the hard cases."""
    if mode == "beta0":
        inp["b"].fill_(-30.0)
    elif mode == "beta1":
        inp["b"].fill_(30.0)
    elif mode == "fast_decay":
        # per-token log-decay down to about -60: in-chunk spans far beyond fp32's exp range
        inp["A_log"].fill_(3.0)
        inp["f"].mul_(3.0).add_(1.0)
    elif mode == "mixed_span":
        # 16-token decay spans around the 80-nat guard: some diagonal blocks factorised,
        # some evaluated pairwise, in the same chunks
        inp["A_log"].fill_(2.0)
        inp["f"].add_(2.0)
    elif mode == "no_decay":
        inp["A_log"].fill_(-30.0)
    return inp


def check_spans(inp, mode):
    """The span cases must really put blocks past the 80-nat guard (so that the
    tensor-core kernels' exact pairwise fallback runs); mixed_span must keep
    others inside it.  Returns the widest span."""
    sp = block_spans(inp)
    wide = float((sp > 80.0).mean())
    if mode == "fast_decay":
        assert wide > 0.5, wide
    elif mode == "mixed_span":
        assert 0.05 < wide < 0.95, wide
    print(f"\n[spans] {mode}: widest {sp.max():.1f} nats, {100 * wide:.0f}% of blocks past 80")
    return float(sp.max())


@pytest.mark.parametrize("mode", ["beta0", "beta1", "fast_decay", "mixed_span", "no_decay"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_degenerate_gates(mode, dtype):
    """Saturated beta, extreme and absent decay, fwd+bwd against the oracle.
    bf16 at 32/64 runs the tensor-core kernels (fwd_chunk, fwd_state,
    bwd_scan, bwd_grad, bwd_gate); fp32 runs the general kernels."""
    w = custom(2, 192, 2, 32, 64, dtype=dtype, h0=True, dh_final=True)
    inp = degenerate(make_inputs(w, seed=13), mode)
    check_spans(inp, mode)
    gpu = run_gpu(inp, True)
    for n, v in gpu.items():
        assert np.isfinite(v).all(), n
    ref = run_oracle(inp, True)
    _report(f"{mode}/{dtype}", compare(gpu, ref, True, bf16=dtype == "bf16"))


@pytest.mark.parametrize("mode", ["fast_decay", "mixed_span"])
def test_span_fallback_packed_documents(mode):
    """The guarded factorisation and its exact pairwise fallback on packed
    documents with one-token, empty and partial chunks (bf16, 32/64)."""
    w = custom(1, 400, 3, 32, 64, dtype="bf16", h0=True, dh_final=True)
    inp = degenerate(make_inputs(w, seed=17, lengths=[1, 0, 70, 17, 64, 1, 200, 47]), mode)
    check_spans(inp, mode)
    gpu = run_gpu(inp, True)
    ref = run_oracle(inp, True)
    _report(f"packed {mode}", compare(gpu, ref, True))


def test_device_only_bad_offsets_flagged():
    """Offsets that exist only on the device are checked by the device: the
    call does no work and kda_device_status reports KDA_ERR_BAD_SEQLENS."""
    from kimi_delta_attention_bwd_gb300 import _lib, kda_device_status
    B, T, H, dk, dv = 1, 128, 2, 32, 64
    dev = "cuda"
    q = torch.randn(B, T, H, dk, device=dev, dtype=torch.bfloat16)
    v = torch.randn(B, T, H, dv, device=dev, dtype=torch.bfloat16)
    b = torch.randn(B, T, H, device=dev, dtype=torch.bfloat16)
    A = torch.zeros(H, device=dev)
    dtb = torch.zeros(H, dk, device=dev)
    cu = torch.tensor([0, 100, 50, 128], dtype=torch.int32, device=dev)  # decreasing
    prob = _lib.make_problem(B, T, H, dk, dv, torch.bfloat16, None, cu, None)
    ws = _lib.alloc_workspace(prob, True)
    o = torch.full((B, T, H, dv), 7.0, device=dev, dtype=torch.bfloat16)
    _lib.kda_fwd(prob, q, q, v, q, b, A, dtb, None, o, None, True, ws)
    assert kda_device_status(ws) == -4
    assert torch.all(o == 7.0)  # nothing written
    good = torch.tensor([0, 50, 100, 128], dtype=torch.int32, device=dev)
    prob2 = _lib.make_problem(B, T, H, dk, dv, torch.bfloat16, None, good, None)
    _lib.kda_fwd(prob2, q, q, v, q, b, A, dtb, None, o, None, True, ws)
    assert kda_device_status(ws) == 0


@pytest.mark.parametrize("dk,dv", [(32, 64), (128, 128)])
def test_deterministic_repeat(dk, dv):
    """Two runs on the same inputs give the same bits (every sum in a fixed
    order, no atomics), on the tensor-core and on the large-head kernels."""
    inp = make_inputs(custom(2, 300, 4, dk, dv, dtype="bf16", h0=True, dh_final=True), seed=14)
    a = run_gpu(inp, True)
    b = run_gpu(inp, True)
    for n in a:
        assert np.array_equal(a[n], b[n]), n
