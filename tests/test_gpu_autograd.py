"""The torch.autograd forms (kimi_delta_attention_bwd_gb300.autograd) give
the outputs and, through loss.backward(), the gradients of the direct calls,
bit for bit: they marshal the same library calls."""
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import (gated_norm, kda_attention, kda_backward, kda_forward,
                                            kda_norm_gate, kda_norm_gate_backward, kda_short_conv,
                                            kda_short_conv_backward, short_conv)
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs, norm_gate_inputs, short_conv_inputs
from _common import to_dev

pytestmark = pytest.mark.gpu

LEAVES = ("q", "k", "v", "f", "b", "A_log", "dt_bias", "h0")
GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "f": "df", "b": "db", "A_log": "dA_log", "dt_bias": "ddt_bias",
           "h0": "dh0"}


@pytest.mark.parametrize("dk,dv", [(32, 64), (128, 128)])
def test_kda_attention_matches_the_direct_calls(dk, dv):
    inp = make_inputs(custom(1, 300, 4, dk, dv, dtype="bf16", h0=True, dh_final=True), seed=41,
                      lengths=[100, 1, 199])
    d = to_dev(inp)
    cu_host = inp["cu_seqlens"].numpy()
    x = {n: d[n].clone().requires_grad_(True) for n in LEAVES}
    o, hf = kda_attention(*(x[n] for n in LEAVES[:7]), scale=d["scale"], h0=x["h0"], cu_seqlens=d["cu_seqlens"],
                          cu_seqlens_host=cu_host, output_final_state=True)
    ((o.float() * d["dO"].float()).sum() + (hf * d["dh_final"]).sum()).backward()
    o2, hf2, ctx = kda_forward(*(d[n] for n in LEAVES[:7]), scale=d["scale"], h0=d["h0"],
                               cu_seqlens=d["cu_seqlens"], cu_seqlens_host=cu_host)
    g = kda_backward(ctx, d["dO"], d["dh_final"])
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(hf, hf2)
    for n in LEAVES:
        assert torch.equal(x[n].grad, g[GRAD_OF[n]]), n


def test_output_only_and_no_initial_state():
    inp = make_inputs(custom(2, 130, 2, 32, 64, dtype="bf16"), seed=42)
    d = to_dev(inp)
    q = d["q"].clone().requires_grad_(True)
    o = kda_attention(q, *(d[n] for n in LEAVES[1:7]), scale=d["scale"])
    (o.float() * d["dO"].float()).sum().backward()
    _, _, ctx = kda_forward(*(d[n] for n in LEAVES[:7]), scale=d["scale"])
    g = kda_backward(ctx, d["dO"], want_dh0=False)
    torch.cuda.synchronize()
    assert torch.equal(q.grad, g["dq"])


def test_short_conv_and_gated_norm_match_the_direct_calls():
    sc = to_dev(short_conv_inputs(300, 192))
    cu = torch.tensor([0, 7, 300], dtype=torch.int32, device="cuda")
    xs, ws = sc["x"].clone().requires_grad_(True), sc["w"].clone().requires_grad_(True)
    y = short_conv(xs, ws, cu)
    (y.float() * sc["dy"].float()).sum().backward()
    dx, dw = kda_short_conv_backward(sc["x"], sc["w"], sc["dy"], cu)
    assert torch.equal(y, kda_short_conv(sc["x"], sc["w"], cu))
    assert torch.equal(xs.grad, dx) and torch.equal(ws.grad, dw)

    ng = to_dev(norm_gate_inputs(200, 64))
    xn, gn, wn = (ng[n].clone().requires_grad_(True) for n in ("x", "g", "w"))
    yn = gated_norm(xn, gn, wn)
    (yn.float() * ng["dy"].float()).sum().backward()
    ex, eg, ew = kda_norm_gate_backward(ng["x"], ng["g"], ng["w"], ng["dy"])
    torch.cuda.synchronize()
    assert torch.equal(yn, kda_norm_gate(ng["x"], ng["g"], ng["w"]))
    assert torch.equal(xn.grad, ex) and torch.equal(gn.grad, eg) and torch.equal(wn.grad, ew)
