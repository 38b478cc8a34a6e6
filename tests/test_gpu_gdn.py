"""Scalar-gated (Gated DeltaNet) variant: one log-decay per token and head,
broadcast over the key channels (f [.., H], dt_bias [H]).

The oracle runs the same recurrence with f and dt_bias repeated over dk and
sums the gate gradients over the channels (tests/_common.run_oracle)."""
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_decode_step
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import TOL_IO, TOL_STATE, compare, rel_fro, rel_max, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    ("fast path bf16 32/64", custom(2, 300, 4, 32, 64, dtype="bf16", h0=True, dh_final=True, gate="scalar"), None),
    ("fast path varlen", custom(1, 300, 4, 32, 64, dtype="bf16", h0=True, dh_final=True, gate="scalar"),
     [1, 0, 130, 64, 105]),
    ("general path fp32 32/64", custom(1, 200, 2, 32, 64, dtype="f32", h0=True, dh_final=True, gate="scalar"), None),
    ("general path bf16 64/128", custom(1, 150, 2, 64, 128, dtype="bf16", dh_final=True, gate="scalar"), None),
    ("general path bf16 128/128 varlen", custom(1, 200, 2, 128, 128, dtype="bf16", h0=True, dh_final=True,
                                                 gate="scalar"), [70, 1, 129]),
]


@pytest.mark.parametrize("name,w,lens", CASES, ids=[c[0] for c in CASES])
def test_gdn_fwd_bwd_matches_oracle(name, w, lens):
    inp = make_inputs(w, seed=91, lengths=lens)
    assert inp["f"].dim() == 3 and inp["dt_bias"].dim() == 1
    gpu = run_gpu(inp, backward=True)
    ref = run_oracle(inp, backward=True)
    errs = compare(gpu, ref, backward=True, bf16=(w.dtype == "bf16"))
    print(f"[gdn] {name}: " + ", ".join(f"{k}={v:.2e}" for k, v in errs.items()))


def test_gdn_decode_matches_oracle():
    n, H, T, dk, dv = 4, 3, 3, 32, 64
    inp = make_inputs(custom(n, T, H, dk, dv, dtype="bf16", h0=True, gate="scalar"), seed=92, with_grad_inputs=False)
    ref = run_oracle(inp, backward=False)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = d["h0"].clone()
    outs = []
    for t in range(T):
        outs.append(kda_decode_step(*(d[x][:, t].contiguous() for x in ("q", "k", "v", "f", "b")), d["A_log"],
                                    d["dt_bias"], state, scale=d["scale"]))
    torch.cuda.synchronize()
    o = torch.stack(outs, 1).double().cpu().numpy().reshape(n * T, H, dv)
    assert rel_max(o, ref["o"], bf16=True) <= TOL_IO
    assert rel_fro(state.cpu().numpy(), ref["h_final"]) <= TOL_STATE
