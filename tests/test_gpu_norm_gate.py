"""Gated RMSNorm epilogue (kda_norm_gate_fwd / _bwd) against its oracle, and
the composed KDA -> gated norm forward and backward against the two oracles."""
import numpy as np
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_backward, kda_forward, kda_norm_gate, kda_norm_gate_backward
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs, norm_gate_inputs, numpy_f64
from oracle import norm_gate as ong
from _common import TOL_IO, TOL_STATE, rel_max, rel_rms, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,dv,dt", [(19200, 64, "bf16"), (1001, 64, "bf16"), (777, 128, "f32"), (4099, 128, "bf16")])
def test_norm_gate_matches_oracle(n, dv, dt):
    inp = norm_gate_inputs(n, dv, dt, seed=7 + n)
    d = {k: v.cuda() for k, v in inp.items()}
    y = kda_norm_gate(d["x"], d["g"], d["w"])
    dx, dg, dw = kda_norm_gate_backward(d["x"], d["g"], d["w"], d["dy"])
    torch.cuda.synchronize()
    f64 = {k: v.double().numpy() for k, v in inp.items()}
    ry = ong.forward(f64["x"], f64["g"], f64["w"])
    rdx, rdg, rdw = ong.backward(f64["x"], f64["g"], f64["w"], f64["dy"])
    bf = dt == "bf16"
    for a, r in ((y, ry), (dx, rdx), (dg, rdg)):
        a = a.double().cpu().numpy()
        assert rel_max(a, r, bf16=bf) <= TOL_IO
        if bf:
            assert rel_rms(a, r) <= 5e-3
    assert rel_max(dw.cpu().numpy(), rdw, bf16=False) <= TOL_IO


def test_norm_gate_is_deterministic():
    inp = norm_gate_inputs(5000, 64, "bf16", seed=3)
    d = {k: v.cuda() for k, v in inp.items()}
    r1 = kda_norm_gate_backward(d["x"], d["g"], d["w"], d["dy"])
    r2 = kda_norm_gate_backward(d["x"], d["g"], d["w"], d["dy"])
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_kda_with_gated_norm_composed():
    # y = norm_gate(kda(q, k, v, f, b), gate, w); loss = sum(y * dy)
    w_ = custom(1, 200, 2, 32, 64, dtype="bf16", h0=True)
    inp = make_inputs(w_, seed=61, with_grad_inputs=True)
    ng = norm_gate_inputs(200 * 2, 64, "bf16", seed=62)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    gate = ng["g"].reshape(1, 200, 2, 64).cuda()
    dy = ng["dy"].reshape(1, 200, 2, 64).cuda()
    wt = ng["w"].cuda()
    o, hf, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"], scale=d["scale"],
                             h0=d["h0"])
    y = kda_norm_gate(o, gate, wt)
    do, dgate, dw = kda_norm_gate_backward(o, gate, wt, dy)
    g = kda_backward(ctx, do)
    torch.cuda.synchronize()
    # oracles: the KDA oracle forward, the norm oracle on its (bf16-rounded, as on the device) output
    ref = run_oracle(inp, backward=False)
    o_bf = torch.from_numpy(ref["o"]).to(torch.bfloat16).double().numpy().reshape(400, 64)
    gt, dyt = ng["g"].double().numpy(), ng["dy"].double().numpy()
    ry = ong.forward(o_bf, gt, ng["w"].double().numpy())
    rdo, rdg, rdw = ong.backward(o_bf, gt, ng["w"].double().numpy(), dyt)
    assert rel_max(y.double().cpu().numpy().reshape(400, 64), ry, bf16=True) <= TOL_IO
    assert rel_max(dgate.double().cpu().numpy().reshape(400, 64), rdg, bf16=True) <= TOL_IO
    assert rel_max(dw.cpu().numpy(), rdw, bf16=False) <= TOL_IO
    inp2 = dict(inp)
    inp2["dO"] = torch.from_numpy(rdo.reshape(1, 200, 2, 64)).to(torch.bfloat16)
    ref2 = run_oracle(inp2, backward=True)
    for name in ("dq", "dk", "dv", "df", "db"):
        a = g[name].double().cpu().numpy().reshape(ref2[name].shape)
        assert rel_max(a, ref2[name], bf16=True) <= TOL_IO, name
    assert rel_max(g["dA_log"].cpu().numpy(), ref2["dA_log"], bf16=False) <= TOL_IO
