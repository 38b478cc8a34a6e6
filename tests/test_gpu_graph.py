"""A forward + backward captured in a CUDA graph and replayed gives the same
bits as the same calls launched eagerly, also after new values are copied into
the captured input buffers (the graph holds pointers and sizes only), for
equal-length rows and for packed documents.  The C entry points issue nothing
but kernel launches on the caller's stream, so the whole call is capturable;
the dependent (programmatic) launches become graph edges."""
import pytest
import torch

from kimi_delta_attention_bwd_gb300 import kda_backward, kda_forward
from kimi_delta_attention_bwd_gb300.inputs import custom, make_inputs
from _common import to_dev

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "f", "b", "A_log", "dt_bias", "dO", "h0", "dh_final")


def _call(d, cu_host):
    o, hf, ctx = kda_forward(d["q"], d["k"], d["v"], d["f"], d["b"], d["A_log"], d["dt_bias"],
                             scale=d["scale"], h0=d.get("h0"), cu_seqlens=d.get("cu_seqlens"),
                             cu_seqlens_host=cu_host)
    g = kda_backward(ctx, d["dO"], d.get("dh_final"))
    out = {"o": o, "h_final": hf}
    out.update({k: v for k, v in g.items() if v is not None})
    return out


@pytest.mark.parametrize("case", ["rows", "docs"])
def test_graph_replay_matches_eager(case):
    if case == "rows":
        w, lens = custom(4, 384, 8, 32, 64, dtype="bf16", h0=True, dh_final=True), None
    else:
        w, lens = custom(1, 1000, 8, 32, 64, dtype="bf16", h0=True, dh_final=True), [130, 1, 64, 500, 305]
    first = to_dev(make_inputs(w, seed=31, lengths=lens))
    second = to_dev(make_inputs(w, seed=32, lengths=lens))
    cu_host = None if lens is None else first["cu_seqlens"].cpu().numpy()

    static = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in first.items()}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            _call(static, cu_host)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = _call(static, cu_host)

    for src in (first, second):
        for k in NAMES:
            if isinstance(src.get(k), torch.Tensor):
                static[k].copy_(src[k])
        graph.replay()
        eager = _call(src, cu_host)
        torch.cuda.synchronize()
        for k, v in eager.items():
            assert torch.equal(captured[k], v), k


def test_graph_replay_of_decode_norm_and_conv():
    """Two chained decode steps, the gated norm and the short convolution
    (forward and backward each) captured together and replayed: the same bits
    as the eager calls, the decode state included."""
    from kimi_delta_attention_bwd_gb300 import (kda_decode_step, kda_norm_gate, kda_norm_gate_backward,
                                                kda_short_conv, kda_short_conv_backward)
    from kimi_delta_attention_bwd_gb300.inputs import norm_gate_inputs, short_conv_inputs

    inp = to_dev(make_inputs(custom(6, 2, 4, 32, 64, dtype="bf16", h0=True), seed=33, with_grad_inputs=False))
    ng = to_dev(norm_gate_inputs(300, 64))
    sc = to_dev(short_conv_inputs(500, 192))
    cu = torch.tensor([0, 7, 8, 300, 500], dtype=torch.int32, device="cuda")

    def calls(state):
        outs = {}
        for t in range(2):
            sl = lambda x: x[:, t].contiguous()  # noqa: E731
            outs[f"o{t}"] = kda_decode_step(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["f"]), sl(inp["b"]),
                                            inp["A_log"], inp["dt_bias"], state, scale=inp["scale"])
        outs["state"] = state
        outs["y"] = kda_norm_gate(ng["x"], ng["g"], ng["w"])
        outs["dx"], outs["dg"], outs["dw"] = kda_norm_gate_backward(ng["x"], ng["g"], ng["w"], ng["dy"])
        outs["cy"] = kda_short_conv(sc["x"], sc["w"], cu)
        outs["cdx"], outs["cdw"] = kda_short_conv_backward(sc["x"], sc["w"], sc["dy"], cu)
        return outs

    state_g = inp["h0"].clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls(inp["h0"].clone())
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = calls(state_g)
    state_g.copy_(inp["h0"])  # capture launched nothing: start the replay from h0
    graph.replay()
    eager = calls(inp["h0"].clone())
    torch.cuda.synchronize()
    for k, v in eager.items():
        assert torch.equal(captured[k], v), k
