"""GPU parity of the whole layer forward against the float64 oracle.

(c) with bf16 inputs and fp32 accumulation, max |err| <= 2e-2 * RMS(y_ref)
and mean |err| <= 2e-3 * RMS(y_ref).  Small and mid-size shapes are compared
on every token (several tiles plus ragged tails); the five full-size layers in
the benchmark's launch configuration are compared on sampled tokens that the
oracle computes one by one.
"""

import numpy as np
import pytest
import torch

import top_routing_expert_gate_b300 as moe
from oracle import moe_oracle as O
from workloads import SHAPES, MoEShape, make_inputs
from workloads.generate import to_f64

from gpu_util import (MARGIN, WEIGHT_REL_SHARED, assert_capacity_layer_close,
                      assert_layer_close, assert_routing_bit_exact, check_tokens,
                      library_routing, np_f, np_i, oracle_layer, oracle_route, same_sets,
                      score_margins)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run_layer(shape, inputs, out_dtype="fp32", ws=None):
    cfg = moe.config_from_shape(shape, out_dtype=out_dtype, T=inputs["x"].shape[0])
    out = moe.layer_forward(cfg, inputs["x"], moe.LayerWeights.from_inputs(inputs), ws=ws)
    torch.cuda.synchronize()
    return cfg, out


def _shape(**kw):
    base = dict(name="custom", T=300, d=256, E=8, k=2, F=384, F_s=0, gate="softmax",
                renormalize=True, rsf=1.0, capacity_factor=None, zipf_s=None, dtype="bf16")
    base.update(kw)
    return MoEShape(**base)


MID_SHAPES = {
    "tiny": SHAPES["tiny"],
    "mid_softmax": _shape(),
    "mid_sigmoid_shared": _shape(T=257, d=192, E=16, k=4, F=256, F_s=384, gate="sigmoid",
                                 rsf=2.5),
    "mid_capacity_zipf": _shape(T=999, d=128, E=8, k=1, F=256, renormalize=False,
                                capacity_factor=1.25, zipf_s=1.2),
    # top-2 with a capacity: second choices compete for slots with later
    # tokens' first choices; several row tiles per expert, a shared expert
    "mid_capacity_k2": _shape(T=1200, d=256, E=8, k=2, F=256, F_s=128, capacity_factor=2.0,
                              zipf_s=1.2),
    "mid_many_experts": _shape(T=129, d=128, E=64, k=6, F=128, F_s=128, gate="sigmoid",
                               rsf=2.5),
    "mid_fp32_shared": _shape(T=77, d=64, E=5, k=3, F=96, F_s=32, dtype="fp32"),
    "single_token": _shape(T=1, d=128, E=4, k=2, F=128),
    "k_equals_E": _shape(T=65, d=64, E=4, k=4, F=128),
    "one_expert_dense": _shape(T=130, d=64, E=1, k=1, F=256),
    # several 128-row M tiles per expert, a ragged last tile, and a down-proj
    # N tail (d = 320 is one full 256-column tile plus 64 columns)
    "mid_multi_mtile": _shape(T=1000, d=320, E=4, k=2, F=256, F_s=128),
    "mid_wide_ff": _shape(T=520, d=128, E=3, k=1, F=1024, gate="sigmoid", rsf=2.5),
    # 257..288 rows in one group: the weights-in-M kernel runs such a tile as
    # two MMAs over both tensor-memory accumulators (every routed expert and
    # the shared expert here; the second shape sits on the 288-row edge with a
    # down-projection N tail)
    "mid_big_tiles": _shape(T=270, d=256, E=2, k=2, F=256, F_s=128, gate="sigmoid", rsf=2.5),
    "mid_big_tile_edge": _shape(T=288, d=320, E=3, k=3, F=128, F_s=128),
    # the shared expert behind a per-token sigmoid gate
    "mid_gated_shared": _shape(T=333, d=256, E=16, k=4, F=256, F_s=256, gate="sigmoid",
                               rsf=2.5, shared_gate=True),
}


def _layer_and_routing(s, inp, ws=None):
    """The fused layer call and, on the same workspace, the split routing
    entry points that expose the fp32 logits and the dispatch arrays."""
    cfg = moe.config_from_shape(s, T=inp["x"].shape[0])
    ws = ws or moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    lib = library_routing(cfg, inp, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(lib["topk_idx"], out["topk_idx"])
    return cfg, out, lib


# the bf16 grouped GEMMs: tokens in the MMA's M (default; a partial token
# tile runs transposed), the same with partial tiles run like full ones, and
# the expert weights in M on CTA pairs
LAYOUTS = ["tokens_m", "tokens_m_full_tail", "weights_m"]


def _set_layout(monkeypatch, layout):
    monkeypatch.setenv("MOE_B300_EXPERT_LAYOUT", layout.replace("_full_tail", ""))
    if layout.endswith("_full_tail"):
        monkeypatch.setenv("MOE_B300_PARTIAL_TILE", "full")
    else:
        monkeypatch.delenv("MOE_B300_PARTIAL_TILE", raising=False)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("name", list(MID_SHAPES))
def test_layer_matches_oracle_all_tokens(name, layout, monkeypatch):
    # every tile layout of the bf16 grouped GEMMs.  The oracle routes from the
    # library's fp32 logits, so (a) the routing and dispatch arrays must agree
    # bit for bit and (c) the output is compared on every token, capacity
    # layers included.
    _set_layout(monkeypatch, layout)
    s = MID_SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=1)
    cfg, out, lib = _layer_and_routing(s, inp)
    ref = oracle_layer(s, inp, logits=np_f(lib["logits"]))
    assert_routing_bit_exact(lib, ref, s.T, s.k)
    np.testing.assert_array_equal(np_i(out["counts"]), ref["counts"])
    np.testing.assert_array_equal(np_i(out["drops"]), ref["drops"])
    np.testing.assert_allclose(np_f(out["topk_w"]), ref["topk_w"], rtol=WEIGHT_REL_SHARED,
                               atol=2e-7)
    if s.capacity_factor is None:
        assert_layer_close(np_f(out["y"]), ref["y"], name)
    else:
        assert ref["drops"].sum() > 0, "the capacity shape must drop assignments"
        assert_capacity_layer_close(np_f(out["y"]), ref["y"], ref["drop_mask"], name)
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], atol=1e-4)


@pytest.mark.parametrize("name", list(MID_SHAPES))
def test_layer_end_to_end_routing(name):
    # (b) the oracle computes its own float64 logits: every token whose
    # k-th/(k+1)-th score margin exceeds 1e-3 chooses the same experts, and
    # (without a capacity, where one flipped token cannot move other tokens'
    # slots) the output of every token with the same chosen set is within
    # the layer tolerance
    s = MID_SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=1)
    cfg, out, lib = _layer_and_routing(s, inp)
    ref = oracle_layer(s, inp)
    margins = score_margins(ref["scores"], ref["topk_idx"])
    same = same_sets(np_i(out["topk_idx"]), ref["topk_idx"])
    assert np.all(same[margins > MARGIN])
    assert same.mean() > 0.9
    np.testing.assert_array_equal(np_i(out["counts"]) + np_i(out["drops"]),
                                  np.bincount(np_i(out["topk_idx"]).ravel(), minlength=s.E))
    if s.capacity_factor is None:
        assert_layer_close(np_f(out["y"])[same], ref["y"][same], name)
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], atol=1e-4)


def test_bf16_output_dtype():
    s = MID_SHAPES["mid_softmax"]
    inp = make_inputs(s, device=DEV, seed=2)
    _, o32 = _run_layer(s, inp, "fp32")
    _, o16 = _run_layer(s, inp, "bf16")
    assert o16["y"].dtype == torch.bfloat16
    torch.testing.assert_close(o16["y"].float(), o32["y"].to(torch.bfloat16).float(),
                               rtol=0, atol=0)


def test_capacity_zero_gives_shared_only():
    s = _shape(T=64, d=128, E=4, k=2, F=128, F_s=128)
    inp = make_inputs(s, device=DEV, seed=3)
    cfg = moe.config_from_shape(s)
    cfg.capacity = 0
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp))
    torch.cuda.synchronize()
    assert out["counts"].sum().item() == 0
    assert out["drops"].sum().item() == 64 * 2
    shared = O.swiglu_ffn(to_f64(inp["x"]), to_f64(inp["ws_gate"]), to_f64(inp["ws_up"]),
                          to_f64(inp["ws_down"]))
    assert_layer_close(np_f(out["y"]), shared, "shared only")
    cfg2 = moe.config_from_shape(_shape(T=64, d=128, E=4, k=2, F=128))
    cfg2.capacity = 0
    inp2 = make_inputs(_shape(T=64, d=128, E=4, k=2, F=128), device=DEV, seed=3)
    out2 = moe.layer_forward(cfg2, inp2["x"], moe.LayerWeights.from_inputs(inp2))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out2["y"]).item() == 0


def test_identical_experts_weight_sum():
    # With every expert identical, y = (sum of routed weights) * FFN(x) + S(x)
    s = _shape(T=200, d=128, E=16, k=4, F=256, F_s=128, gate="sigmoid", rsf=2.5)
    inp = make_inputs(s, device=DEV, seed=4)
    for key in ("w_gate", "w_up", "w_down"):
        inp[key][:] = inp[key][0:1].clone()
    _, out = _run_layer(s, inp)
    x = to_f64(inp["x"])
    ffn = O.swiglu_ffn(x, to_f64(inp["w_gate"][0]), to_f64(inp["w_up"][0]),
                       to_f64(inp["w_down"][0]))
    sh = O.swiglu_ffn(x, to_f64(inp["ws_gate"]), to_f64(inp["ws_up"]), to_f64(inp["ws_down"]))
    assert_layer_close(np_f(out["y"]), 2.5 * ffn + sh, "identical experts")


def test_empty_batch():
    s = _shape(T=0)
    cfg = moe.config_from_shape(s)
    inp = make_inputs(_shape(T=1), device=DEV, seed=5)
    y = torch.empty((0, s.d), dtype=torch.float32, device=DEV)
    x = inp["x"][:0]
    out = moe.layer_forward(cfg, x, moe.LayerWeights.from_inputs(inp), y=y)
    torch.cuda.synchronize()
    assert out["counts"].sum().item() == 0 and out["mean_prob"].abs().sum().item() == 0


def test_deterministic_and_split_calls_match_fused():
    s = MID_SHAPES["mid_sigmoid_shared"]
    inp = make_inputs(s, device=DEV, seed=6)
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    w = moe.LayerWeights.from_inputs(inp)
    a = moe.layer_forward(cfg, inp["x"], w, ws=ws)
    b = moe.layer_forward(cfg, inp["x"], w, ws=ws)
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], b[key]), key
    # the same layer through the separate entry points
    r = moe.route(cfg, inp["x"], w.w_router, w.router_bias, ws=ws)
    dsp = moe.dispatch(cfg, r["topk_idx"], ws=ws)
    A = s.T * s.k
    y_perm = torch.empty((A, s.d), dtype=torch.float32, device=DEV)
    y_sh = torch.empty((s.T, s.d), dtype=torch.float32, device=DEV)
    moe.moe_grouped_swiglu(cfg, inp["x"], dsp["perm"], dsp["offsets"], w.w_gate, w.w_up,
                           w.w_down, w.ws_gate, w.ws_up, w.ws_down, y_perm, y_sh, ws)
    y = torch.empty((s.T, s.d), dtype=torch.float32, device=DEV)
    moe.moe_combine(cfg, y_perm, r["topk_w"], dsp["offsets"], dsp["perm"], dsp["drop_mask"],
                    y_sh, None, y, ws)
    torch.cuda.synchronize()
    assert torch.equal(r["topk_idx"], a["topk_idx"])
    assert torch.equal(y, a["y"])
    assert moe.moe_get_error(ws) == 0


@pytest.mark.parametrize("out_dtype", ["fp32", "bf16"])
def test_host_buffer_call_matches_device_call(out_dtype):
    # the host-buffer entry point: x copied in, the layer, y copied out, on
    # two streams with their own staging buffers and workspaces
    s = MID_SHAPES["mid_sigmoid_shared"]
    inp = make_inputs(s, device=DEV, seed=16)
    cfg = moe.config_from_shape(s, out_dtype=out_dtype)
    w = moe.LayerWeights.from_inputs(inp)
    ref = moe.layer_forward(cfg, inp["x"], w)["y"].cpu()
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = []
    for j in range(4):
        st = streams[j % 2]
        x_host = inp["x"].cpu().pin_memory()
        y_host = torch.full(ref.shape, float("nan"), dtype=ref.dtype).pin_memory()
        x_dev = torch.empty_like(inp["x"])
        y_dev = torch.empty(ref.shape, dtype=ref.dtype, device=DEV)
        ws = moe.Workspace(cfg)
        torch.cuda.synchronize()
        moe.layer_forward_host(cfg, x_host, w, ws, x_dev, y_dev, y_host, stream=st)
        outs.append((y_host, ws))
    torch.cuda.synchronize()
    for y_host, ws in outs:
        assert moe.moe_get_error(ws) == 0
        assert torch.equal(y_host, ref)
    # an empty batch copies nothing
    c0 = moe.config_from_shape(_shape(T=0))
    e = torch.empty((0, s.d), dtype=torch.float32)
    moe.layer_forward_host(c0, e, moe.LayerWeights.from_inputs(make_inputs(_shape(T=1), device=DEV,
                                                                           seed=5)),
                           moe.Workspace(c0), torch.empty((0, s.d), device=DEV),
                           torch.empty((0, s.d), device=DEV), e)
    torch.cuda.synchronize()


def test_gated_shared_expert_split_calls_match_fused():
    s = MID_SHAPES["mid_gated_shared"]
    inp = make_inputs(s, device=DEV, seed=7)
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    w = moe.LayerWeights.from_inputs(inp)
    a = moe.layer_forward(cfg, inp["x"], w, ws=ws)
    r = moe.route(cfg, inp["x"], w.w_router, w.router_bias, ws=ws)
    dsp = moe.dispatch(cfg, r["topk_idx"], ws=ws)
    A = s.T * s.k
    y_perm = torch.empty((A, s.d), dtype=torch.float32, device=DEV)
    y_sh = torch.empty((s.T, s.d), dtype=torch.float32, device=DEV)
    moe.moe_grouped_swiglu(cfg, inp["x"], dsp["perm"], dsp["offsets"], w.w_gate, w.w_up,
                           w.w_down, w.ws_gate, w.ws_up, w.ws_down, y_perm, y_sh, ws)
    gate_w = torch.empty(s.T, dtype=torch.float32, device=DEV)
    moe.moe_shared_gate_weights(cfg, inp["x"], w.shared_gate, gate_w)
    y = torch.empty((s.T, s.d), dtype=torch.float32, device=DEV)
    moe.moe_combine(cfg, y_perm, r["topk_w"], dsp["offsets"], dsp["perm"], dsp["drop_mask"],
                    y_sh, gate_w, y, ws)
    torch.cuda.synchronize()
    assert torch.equal(y, a["y"])
    # the gate weights themselves: sigmoid(x . w), fp32 accumulation of d bf16 products
    want = O.shared_gate_weights(to_f64(inp["x"]), to_f64(w.shared_gate))
    np.testing.assert_allclose(np_f(gate_w), want, rtol=0, atol=2e-6)
    assert moe.moe_get_error(ws) == 0


@pytest.mark.parametrize("counts,drops,P,want", [
    ([2, 2, 2, 2], [0, 0, 0, 0], [0.25, 0.25, 0.25, 0.25], 1.0),
    ([5, 1, 1, 1], [0, 0, 0, 0], [0.55, 0.15, 0.15, 0.15], 1.6),
    ([3, 1, 1, 1], [2, 0, 0, 0], [0.55, 0.15, 0.15, 0.15], 1.6),
    ([8, 0, 0, 0], [0, 0, 0, 0], [1.0, 0.0, 0.0, 0.0], 4.0),
])
def test_balance_loss_worked_values_on_gpu(counts, drops, P, want):
    # "辅助损失": N * sum f P = 1.0 uniform, 1.6 skewed, 4.0 collapsed (alpha = 0.01)
    cfg = moe.make_config(8, 64, 4, 1, 128, act_dtype="fp32")
    loss = torch.zeros(1, dtype=torch.float32, device=DEV)
    moe.moe_balance_loss(cfg, torch.tensor(counts, dtype=torch.int32, device=DEV),
                         torch.tensor(drops, dtype=torch.int32, device=DEV),
                         torch.tensor(P, dtype=torch.float32, device=DEV), 0.01, loss)
    torch.cuda.synchronize()
    assert loss.item() == pytest.approx(0.01 * want, rel=1e-6)


def test_balance_loss_from_layer_statistics():
    s = MID_SHAPES["mid_capacity_zipf"]
    inp = make_inputs(s, device=DEV, seed=8)
    cfg = moe.config_from_shape(s)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp))
    loss = torch.zeros(1, dtype=torch.float32, device=DEV)
    moe.moe_balance_loss(cfg, out["counts"], out["drops"], out["mean_prob"], 0.02, loss)
    torch.cuda.synchronize()
    want = O.balance_loss(np_i(out["counts"]), np_i(out["drops"]), np_f(out["mean_prob"]), 0.02)
    assert loss.item() == pytest.approx(want, rel=1e-6)
    assert loss.item() > 0.02   # the Zipf skew makes it exceed the balanced minimum alpha


# ---------------------------------------------------------------------------
# The five full-size layers, in the benchmark's launch configuration
# ---------------------------------------------------------------------------

FULL = ["tiny", "mixtral", "dsv3_prefill", "switch", "dsv3_decode"]
# tokens whose outputs the oracle computes at full size (all of them for the
# small batches); each expert's ragged last row tile is always among them
FULL_CHECK = {"tiny": 64, "mixtral": 64, "dsv3_prefill": 320, "switch": 96, "dsv3_decode": 64}


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_layer_sampled(name):
    s = SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=0)
    cfg, out, lib = _layer_and_routing(s, inp)
    # (a) from the library's fp32 logits: routing and dispatch bit for bit
    ref = oracle_route(s, np_f(lib["logits"]))
    assert_routing_bit_exact(lib, ref, s.T, s.k)
    np.testing.assert_array_equal(np_i(out["counts"]), ref["counts"])
    np.testing.assert_array_equal(np_i(out["drops"]), ref["drops"])
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], atol=1e-4)
    # (b) end to end: margin-clear tokens choose the same experts
    z = O.router_logits(to_f64(inp["x"]), to_f64(inp["w_router"]), to_f64(inp["router_bias"]))
    ref_b = oracle_route(s, z)
    same = same_sets(np_i(out["topk_idx"]), ref_b["topk_idx"])
    assert np.all(same[score_margins(ref_b["scores"], ref_b["topk_idx"]) > MARGIN])
    assert same.mean() > 0.97
    # (c) outputs: every expert's ragged-tail token, the shared expert's first
    # and last tiles, dropped tokens, random ones
    pick = check_tokens(ref, s.T, s.k, FULL_CHECK[name])
    assert len(pick) >= min(FULL_CHECK[name], s.T)
    oref = oracle_layer(s, inp, tokens=pick, logits=np_f(lib["logits"]))
    y = np_f(out["y"])[pick]
    if s.capacity_factor is None:
        assert_layer_close(y, oref["y"], name)
    else:
        dm = ref["drop_mask"].reshape(s.T, s.k)[pick]
        assert dm.any() and not dm.all()
        assert_capacity_layer_close(y, oref["y"], dm, name)
