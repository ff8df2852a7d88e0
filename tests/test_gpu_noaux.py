"""GPU parity of DeepSeek-V3's auxiliary-loss-free router ("10. 混合专家 MoE：
总参数与激活参数", section "DeepSeek-V3 的无辅助损失偏置"): ranking by s + b with
a selection-only bias, expert groups scored by their two best keys, weights
from the raw scores, and the bias step after a batch.

Fed the same fp32 logits, the kernel ranks by fp32 s + b, so a decision can
differ from the float64 oracle only when it is closer than the rounding of
the sigmoid and the addition.  Every token whose selection margin (k-th chosen
key over the best unchosen key of the kept groups, and the last kept group
over the best dropped group) exceeds KEY_MARGIN must choose the same experts
in the same order; end to end (bf16 inputs) the margin is the routing
margin MARGIN of the other parity tests.
"""

import numpy as np
import pytest
import torch

import top_routing_expert_gate_b300 as moe
from oracle import moe_oracle as O
from workloads import SHAPES, MoEShape, make_inputs
from workloads.generate import to_f64

from gpu_util import (MARGIN, assert_layer_close, biased_margins, check_tokens,
                      library_routing, np_f, np_i, oracle_layer, same_sets)

pytestmark = pytest.mark.gpu

DEV = "cuda"
KEY_MARGIN = 1e-5

CASES = {
    # name: (T, E, k, n_group, topk_group, bias_std, gate)
    "dsv3_groups": (4096, 256, 8, 8, 4, 0.02, "sigmoid"),
    "groups_64": (1000, 64, 6, 8, 3, 0.05, "sigmoid"),
    "softmax_groups": (513, 16, 4, 4, 2, 0.1, "softmax"),
    "bias_no_groups": (300, 32, 2, 0, 0, 0.05, "sigmoid"),
    "groups_no_bias": (300, 32, 4, 4, 2, None, "sigmoid"),
    "one_group_kept": (257, 24, 3, 6, 1, 0.05, "sigmoid"),
}


def _case(name, seed=21):
    T, E, k, ng, tg, std, gate = CASES[name]
    g = torch.Generator().manual_seed(seed)
    z = torch.randn((T, E), generator=g, dtype=torch.float32)
    b = None if std is None else torch.randn(E, generator=g, dtype=torch.float32) * std
    cfg = moe.make_config(T, 64, E, k, 128, gate=gate, renormalize=True, rsf=2.5,
                          act_dtype="fp32", n_group=ng, topk_group=tg)
    return cfg, z, b, (T, E, k, max(ng, 1), tg, gate)


def _ordered(keys_sel: np.ndarray, margin: float) -> np.ndarray:
    """Rows whose consecutive chosen keys are separated by the margin."""
    if keys_sel.shape[1] == 1:
        return np.ones(keys_sel.shape[0], dtype=bool)
    return np.all(keys_sel[:, :-1] - keys_sel[:, 1:] > margin, axis=1)


@pytest.mark.parametrize("name", list(CASES))
def test_biased_grouped_topk_from_logits(name):
    cfg, z, b, (T, E, k, ng, tg, gate) = _case(name)
    out = moe.topk_from_logits(cfg, z.to(DEV), score_bias=None if b is None else b.to(DEV))
    torch.cuda.synchronize()
    z64 = z.double().numpy()
    b64 = None if b is None else b.double().numpy()
    scores = O.gate_scores(z64, gate)
    ref = O.route(z64, k, gate, True, 2.5, None, score_bias=b64, n_group=ng, topk_group=tg)
    gi = np_i(out["topk_idx"])
    m = biased_margins(scores, b64, ref["topk_idx"], ng, tg)
    keys = scores + (0.0 if b64 is None else b64[None, :])
    sel = np.take_along_axis(keys, ref["topk_idx"], axis=1)
    clear = (m > KEY_MARGIN) & _ordered(sel, KEY_MARGIN)
    assert clear.mean() > 0.95
    np.testing.assert_array_equal(gi[clear], ref["topk_idx"][clear])
    same = np.all(gi == ref["topk_idx"], axis=1)
    # weights come from the raw scores of the chosen experts
    np.testing.assert_allclose(np_f(out["topk_w"])[same], ref["topk_w"][same], rtol=2e-6,
                               atol=2e-6)
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], rtol=1e-4, atol=1e-6)
    # every token, ambiguous or not, stays within topk_group groups
    if ng > 1:
        gs = E // ng
        assert all(len(set((gi[t] // gs).tolist())) <= tg for t in range(T))
    assert np.all(np.sort(gi, axis=1)[:, 1:] != np.sort(gi, axis=1)[:, :-1])   # distinct


def test_score_bias_step_matches_oracle():
    rng = np.random.default_rng(3)
    E = 256
    cfg = moe.make_config(1, 64, E, 8, 128, act_dtype="fp32")
    counts = rng.integers(0, 600, size=E).astype(np.int32)
    drops = rng.integers(0, 40, size=E).astype(np.int32)
    counts[:4] = 256   # a few experts exactly at a round load
    b0 = (rng.normal(size=E) * 0.01).astype(np.float32)
    bias = torch.from_numpy(b0.copy()).to(DEV)
    moe.moe_update_score_bias(cfg, torch.from_numpy(counts).to(DEV),
                              torch.from_numpy(drops).to(DEV), 0.001, bias)
    torch.cuda.synchronize()
    want = O.update_score_bias(b0.astype(np.float64), counts + drops, 0.001)
    np.testing.assert_allclose(np_f(bias), want, rtol=0, atol=1e-7)
    # loads all equal: nothing moves, bit for bit
    same = torch.full((E,), 7, dtype=torch.int32, device=DEV)
    before = bias.clone()
    moe.moe_update_score_bias(cfg, same, None, 0.5, bias)
    torch.cuda.synchronize()
    assert torch.equal(before, bias)


def test_printed_bias_trace_replayed_on_gpu(golden):
    # the page's 8-token, 4-expert, top-1 simulation with gamma = 0.05, run
    # through the library: route with the bias, count the loads, step the bias
    fx = golden("moe10_bias_update_trace.json")
    s = torch.tensor(fx["constructed_scores"], dtype=torch.float64)
    z = torch.log(s / (1 - s)).to(torch.float32).to(DEV)    # sigmoid(z) = s
    cfg = moe.make_config(fx["T"], 64, fx["E"], fx["k"], 128, gate="sigmoid",
                          renormalize=False, act_dtype="fp32")
    bias = torch.zeros(fx["E"], dtype=torch.float32, device=DEV)
    ws = moe.Workspace(cfg)
    for step in fx["steps"]:
        np.testing.assert_allclose(np_f(bias), step["bias"], atol=1e-6)
        r = moe.topk_from_logits(cfg, z, ws, score_bias=bias)
        d = moe.dispatch(cfg, r["topk_idx"], ws)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(np_i(d["counts"]), step["load"])
        # the weight is the raw score of the chosen expert, never s + b
        np.testing.assert_allclose(
            np_f(r["topk_w"])[:, 0],
            s.numpy()[np.arange(fx["T"]), np_i(r["topk_idx"])[:, 0]], rtol=1e-6)
        moe.moe_update_score_bias(cfg, d["counts"], d["drops"], fx["gamma"], bias)
    assert moe.moe_get_error(ws) == 0


def _noaux_shape(**kw):
    base = dict(name="noaux", T=300, d=256, E=32, k=4, F=256, F_s=128, gate="sigmoid",
                renormalize=True, rsf=2.5, capacity_factor=None, zipf_s=None, dtype="bf16",
                n_group=4, topk_group=2, score_bias_std=0.05)
    base.update(kw)
    return MoEShape(**base)


def _end_to_end_clear(shape, inp, ref, gi):
    scores = ref["scores"]
    b64 = to_f64(inp["score_bias"])
    m = biased_margins(scores, b64, ref["topk_idx"], max(shape.n_group, 1), shape.topk_group)
    return (m > MARGIN), same_sets(gi, ref["topk_idx"])


@pytest.mark.parametrize("layout", ["tokens_m", "weights_m"])
@pytest.mark.parametrize("kw", [{}, {"T": 129, "E": 64, "k": 8, "n_group": 8, "topk_group": 4},
                                {"n_group": 0, "topk_group": 0}])
def test_layer_noaux_all_tokens(kw, layout, monkeypatch):
    monkeypatch.setenv("MOE_B300_EXPERT_LAYOUT", layout)
    s = _noaux_shape(**kw)
    inp = make_inputs(s, device=DEV, seed=4)
    cfg = moe.config_from_shape(s)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp))
    torch.cuda.synchronize()
    ref = oracle_layer(s, inp)
    gi = np_i(out["topk_idx"])
    clear, same = _end_to_end_clear(s, inp, ref, gi)
    assert np.all(same[clear])
    assert same.mean() > 0.9
    assert_layer_close(np_f(out["y"])[same], ref["y"][same], "noaux layer")
    np.testing.assert_array_equal(np_i(out["counts"]).sum(), s.T * s.k)


@pytest.mark.slow
def test_full_size_dsv3_noaux_sampled():
    s = SHAPES["dsv3_prefill_noaux"]
    inp = make_inputs(s, device=DEV, seed=0)
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    lib = library_routing(cfg, inp, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(lib["topk_idx"], out["topk_idx"])
    gi = np_i(out["topk_idx"])
    b64 = to_f64(inp["score_bias"])
    # from the library's fp32 logits: key-margin-clear tokens choose the same
    # experts in the same order
    zl = np_f(lib["logits"])
    ref = O.route(zl, s.k, s.gate, s.renormalize, s.rsf, None, score_bias=b64,
                  n_group=s.n_group, topk_group=s.topk_group)
    km = biased_margins(ref["scores"], b64, ref["topk_idx"], s.n_group, s.topk_group)
    np.testing.assert_array_equal(gi[km > KEY_MARGIN], ref["topk_idx"][km > KEY_MARGIN])
    # end to end from float64 logits
    z = O.router_logits(to_f64(inp["x"]), to_f64(inp["w_router"]))
    ref_b = O.route(z, s.k, s.gate, s.renormalize, s.rsf, None, score_bias=b64,
                    n_group=s.n_group, topk_group=s.topk_group)
    clear, same_b = _end_to_end_clear(s, inp, ref_b, gi)
    assert np.all(same_b[clear])
    assert same_b.mean() > 0.97
    gs = s.E // s.n_group
    assert all(len(set((gi[t] // gs).tolist())) <= s.topk_group for t in range(s.T))
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], atol=1e-4)
    # outputs of every expert's ragged-tail token (from the library's own
    # dispatch) and random tokens, among those routed like the oracle
    same = same_sets(gi, ref["topk_idx"])
    assert same.mean() > 0.99
    disp = {"offsets": np_i(lib["offsets"]), "perm": np_i(lib["perm"]),
            "drop_mask": np_i(lib["drop_mask"])[: s.T * s.k]}
    pick = check_tokens(disp, s.T, s.k, 320)
    pick = pick[same[pick]]
    assert len(pick) >= 300
    oref = oracle_layer(s, inp, tokens=pick, logits=zl)
    assert_layer_close(np_f(out["y"])[pick], oref["y"], "dsv3 noaux")
