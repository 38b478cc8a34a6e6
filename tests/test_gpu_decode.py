"""Single-token recurrent step (kda_decode) against the oracle.

The oracle is the token-by-token recurrence run on one-token documents whose
initial states are the decode states; chained steps are compared with the
oracle over the same tokens as one document, and the decode step after a
chunked prefill is compared with the chunked forward over one more token.
"""
import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_decode_step, kda_forward
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import TOL_IO, TOL_STATE, rel_fro, rel_max, run_oracle

pytestmark = pytest.mark.gpu

SHAPES = [(32, 64, "bf16"), (32, 64, "f32"), (64, 64, "bf16"), (64, 128, "f32"), (128, 128, "bf16")]


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


@pytest.mark.parametrize("dk,dv,dt", SHAPES)
def test_decode_steps_match_oracle(dk, dv, dt):
    # 5 sequences of 4 tokens; the oracle runs them as 5 documents of 4 tokens
    n, H, T = 5, 3, 4
    inp = make_inputs(custom(n, T, H, dk, dv, dtype=dt, h0=True), seed=31 + dk + dv, with_grad_inputs=False)
    ref = run_oracle(inp, backward=False)
    d = _dev(inp)
    state = d["h0"].clone()
    outs = []
    for t in range(T):
        sl = lambda x: x[:, t].contiguous()  # noqa: E731
        outs.append(kda_decode_step(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["f"]), sl(d["b"]), d["A_log"],
                                    d["dt_bias"], state, scale=d["scale"]))
    torch.cuda.synchronize()
    o = torch.stack(outs, 1).double().cpu().numpy().reshape(n * T, H, dv)  # oracle: flattened tokens
    assert rel_max(o, ref["o"], bf16=(dt == "bf16")) <= TOL_IO
    assert rel_fro(state.cpu().numpy(), ref["h_final"]) <= TOL_STATE


def test_decode_after_prefill_matches_chunked_forward():
    # prefill 77 tokens with the chunked forward, decode token 78; compare with
    # the chunked forward over all 78 tokens (both on the GPU, both against the
    # same recurrence)
    B, T, H, dk, dv = 2, 78, 4, 32, 64
    inp = make_inputs(custom(B, T, H, dk, dv, dtype="bf16", h0=True), seed=57, with_grad_inputs=False)
    d = _dev(inp)
    pre = {k: d[k][:, :T - 1].contiguous() for k in ("q", "k", "v", "f", "b")}
    _, h77, _ = kda_forward(pre["q"], pre["k"], pre["v"], pre["f"], pre["b"], d["A_log"], d["dt_bias"],
                            scale=d["scale"], h0=d["h0"], save_for_backward=False)
    last = {k: d[k][:, T - 1].contiguous() for k in ("q", "k", "v", "f", "b")}
    state = h77.clone()
    o_dec = kda_decode_step(last["q"], last["k"], last["v"], last["f"], last["b"], d["A_log"], d["dt_bias"],
                            state, scale=d["scale"])
    o_all, h78, _ = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], scale=d["scale"],
                                h0=d["h0"], save_for_backward=False)
    torch.cuda.synchronize()
    a = o_dec.double().cpu().numpy()
    r = o_all[:, T - 1].double().cpu().numpy()
    assert rel_max(a, r, bf16=True) <= TOL_IO
    assert rel_fro(state.cpu().numpy(), h78.cpu().numpy()) <= TOL_STATE


def test_decode_rejects_bad_arguments():
    from kimi_delta_attention_bwd_gb300 import _lib
    lib = _lib.load()
    z = torch.zeros(64, device="cuda")
    p = _lib._p
    st = lib.kda_decode(2, 2, 48, 64, 0, 0, 0.0, *([p(z)] * 9), _lib._stream())
    assert st == -2  # unsupported (dk, dv)
    st = lib.kda_decode(0, 2, 32, 64, 0, 0, 0.0, *([p(z)] * 9), _lib._stream())
    assert st == -1
    st = lib.kda_decode(2, 2, 32, 64, 0, 7, 0.0, *([p(z)] * 9), _lib._stream())
    assert st == -1  # unknown gate mode
