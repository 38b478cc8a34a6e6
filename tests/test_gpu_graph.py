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
