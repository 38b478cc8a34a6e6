"""Split state chains of the tensor-core path against the oracle.

The forward state chain S_{c+1} = M_c S_c + KU_c is affine, so a run of chunks
composes into one map S -> Phi S + B; so is the backward's reverse chain
dS_c = M_c^T dS_{c+1} + QW_c^T dO_c (dS -> Psi dS + D).  When a workload's
longest document has more than 32 chunks and more than twice the average
chain length per resident chain CTA (a chain-bound workload, such as one long
document packed with short ones), every document over 32 chunks runs as
segments of 16 chunks: one kernel per direction composes each segment but the
one its chain starts in, and the chain kernels start every other segment from
the composites before it (after it, in the backward) folded onto h0
(dS_final).  The torchtitan PR "[kimi k3] Support sample packing in KDA"
(description: the recurrent state resets at document boundaries) fixes what
a packed document must equal: the same document run alone.

Cases force the split at H = 2 or 1 (a few chains on the whole GPU): a long
document packed with one-token, empty and short ones; long equal rows;
exactly 33 chunks (segments of 16, 16 and 1); the scalar gate; no states; a
301-chunk document (segments of 32 chunks, folds of up to nine).  Forward and
backward (with h0 and dS_final) are compared with the oracle at the parity
tolerances; the grid planned on the host (host copy of cu_seqlens) and on the
device (device-only offsets) give the same bits; a packed long document equals
its separate run bit for bit (a lone document over 32 chunks is always split
the same way); 32 chunks run whole and 33 run split.
"""
import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import _lib, kda_backward, kda_forward
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import compare, run_oracle

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, seed, document lengths)
    "packed_long_doc": (custom(1, 64 * 40 + 17 + 401, 2, 32, 64, h0=True, dh_final=True), 61,
                        [64 * 40 + 17, 100, 1, 0, 300]),
    "rows_51_chunks": (custom(2, 64 * 50 + 5, 2, 32, 64, h0=True, dh_final=True), 62, None),
    "exactly_33_chunks": (custom(1, 64 * 32 + 1, 2, 32, 64, h0=True, dh_final=True), 63, None),
    "scalar_gate_long": (custom(1, 64 * 40 + 30, 2, 32, 64, gate="scalar", h0=True, dh_final=True), 64, None),
    # no initial state and no final-state gradient: the folds start from zero
    "packed_no_states": (custom(1, 64 * 45 + 200, 2, 32, 64), 66, [64 * 45, 150, 50]),
    # 301 chunks: segments of 32 chunks (the least multiple of 16 whose square covers 301), ten of
    # them, folds of up to nine composites
    "very_long_doc": (custom(1, 64 * 300 + 7, 1, 32, 64, h0=True, dh_final=True), 67, None),
}


def _run(inp, host_offsets=True):
    """kda_forward + kda_backward on the device; float64 numpy results in the
    flattened [Ntok, H, ...] layout.  host_offsets=False passes cu_seqlens on
    the device only, so that the device plans the split."""
    dev = "cuda"
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu = d.get("cu_seqlens")
    cu_host = inp["cu_seqlens"].numpy() if (cu is not None and host_offsets) else None
    o, hf, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], scale=d["scale"],
                             h0=d.get("h0"), cu_seqlens=cu, cu_seqlens_host=cu_host)
    g = kda_backward(ctx, d["dO"], d.get("dh_final"))
    torch.cuda.synchronize()
    B, T, H = inp["q"].shape[:3]
    out = {"o": o, "h_final": hf, **g}
    res = {}
    for k, v in out.items():
        if v is None:
            continue
        v = v.detach().to(torch.float64).cpu().numpy()
        if k in ("o", "dq", "dk", "dv", "df", "db"):
            v = v.reshape(B * T, H, *v.shape[3:]) if v.ndim == 4 else v.reshape(B * T, H)
        res[k] = v
    return res


def _launches(fn):
    """{kernel name: launches} of the library's kernels during fn()."""
    _lib.prof_start()
    fn()
    torch.cuda.synchronize()
    return {k: int(v[1]) for k, v in _lib.prof_stop().items() if v[1]}


@pytest.mark.parametrize("name", list(CASES))
def test_split_chain_matches_oracle(name):
    w, seed, lens = CASES[name]
    inp = make_inputs(w, seed=seed, lengths=lens)
    n = _launches(lambda: _run(inp))
    assert n.get("fwd_seg", 0) == 1 and n.get("bwd_seg", 0) == 1, n  # the case is split
    gpu = _run(inp)
    ref = run_oracle(inp, True)
    errs = compare(gpu, ref, True)
    if inp.get("cu_seqlens") is not None:  # the device plans the same split: the same bits
        dev_planned = _run(inp, host_offsets=False)
        for k in gpu:
            assert np.array_equal(gpu[k], dev_planned[k]), k
    print(f"\n[split chain] {name}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))


def test_split_long_doc_equals_separate_bitwise():
    w, seed, lens = CASES["packed_long_doc"]
    inp = make_inputs(w, seed=seed, lengths=lens)
    packed = _run(inp)
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
        one = _run(sub)
        for k in ("o", "dq", "dk", "dv", "df", "db"):
            assert np.array_equal(one[k], packed[k][t0:t1]), (s, k)
        assert np.array_equal(one["h_final"][0], packed["h_final"][s]), s
        assert np.array_equal(one["dh0"][0], packed["dh0"][s]), s


@pytest.mark.parametrize("chunks,split", [(32, False), (33, True)])
def test_split_boundary(chunks, split):
    w = custom(1, 64 * chunks, 2, 32, 64, h0=True)
    inp = make_inputs(w, seed=65, with_grad_inputs=True)
    n = _launches(lambda: _run(inp))
    assert (n.get("fwd_seg", 0) == 1) == split and (n.get("bwd_seg", 0) == 1) == split, n
    assert n.get("fwd_state", 0) == 1 and n.get("bwd_scan", 0) == 1, n
