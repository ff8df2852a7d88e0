"""The layer forward captured in a CUDA graph.

Every step of moe_layer_forward is enqueued on the caller's stream with no
host synchronisation and no allocation, so the whole call can be captured
once and replayed: a replay must read the current contents of the captured
input buffer and give the eager call's output bit for bit.
"""

import pytest
import torch

import top_routing_expert_gate_b300 as moe
from workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _shape(**kw):
    base = dict(name="graph", T=257, d=256, E=16, k=4, F=256, F_s=384, gate="sigmoid",
                renormalize=True, rsf=2.5, capacity_factor=None, zipf_s=None, dtype="bf16")
    base.update(kw)
    return MoEShape(**base)


GRAPH_SHAPES = {
    "bf16_shared": _shape(),
    "bf16_capacity": _shape(T=700, E=8, k=2, F_s=0, gate="softmax", rsf=1.0,
                            capacity_factor=1.0, zipf_s=1.2),
    "fp8_decode": _shape(T=40, d=512, E=32, F_s=256, weight_format="fp8"),
    "expert_choice": _shape(T=512, E=8, k=2, F_s=0, gate="softmax", renormalize=False, rsf=1.0,
                            routing="expert"),
}


@pytest.mark.parametrize("name", list(GRAPH_SHAPES))
def test_layer_forward_replays_from_a_cuda_graph(name):
    s = GRAPH_SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=17)
    cfg = moe.config_from_shape(s)
    w = moe.LayerWeights.from_inputs(inp)
    ws = moe.Workspace(cfg)
    x = inp["x"].clone()
    y = torch.empty((s.T, s.d), dtype=torch.float32, device=DEV)
    # one eager call first (one-time kernel attribute setup stays outside the capture)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        moe.layer_forward(cfg, x, w, ws=ws, y=y, stats=False)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.layer_forward(cfg, x, w, ws=ws, y=y, stats=False)
    torch.cuda.synchronize()

    other = make_inputs(s, device=DEV, seed=18)["x"]
    for src in (inp["x"], other, inp["x"]):
        x.copy_(src)
        graph.replay()
        eager = moe.layer_forward(cfg, src.clone(), w, stats=False)["y"]
        torch.cuda.synchronize()
        assert torch.equal(y, eager)
    assert moe.moe_get_error(ws) == 0
