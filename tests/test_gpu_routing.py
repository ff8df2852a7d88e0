"""GPU parity of routing and dispatch against the float64 oracle.

(a) fed the same fp32 logits, top-k indices, counts, drops, offsets,
    permutation and drop mask are bit-exact;
(b) end to end from x and W_router, every token whose k-th/(k+1)-th score
    margin exceeds 1e-3 routes identically and weights agree within 1e-3.
"""

import numpy as np
import pytest
import torch

import top_routing_expert_gate_b300 as moe
from oracle import moe_oracle as O
from workloads import SHAPES, make_inputs
from workloads.generate import to_f64

from gpu_util import (MARGIN, WEIGHT_ABS, np_f, np_i, oracle_capacity, order_separated,
                      same_sets, score_margins)

pytestmark = pytest.mark.gpu

DEV = "cuda"

# the layers routed by logit top-k (the DeepSeek-V3 score-bias router is
# covered in test_gpu_noaux.py)
LOGIT_SHAPES = [n for n, s in SHAPES.items()
                if s.n_group == 0 and s.score_bias_std is None and s.routing == "token"]


def _logits(T, E, seed, quantize=None):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn((T, E), generator=g, dtype=torch.float32)
    if quantize:
        z = torch.round(z / quantize) * quantize   # forces many exact ties
    return z


def _cfg(shape, T, capacity=None):
    c = moe.config_from_shape(shape, T=T)
    if capacity is not None:
        c.capacity = capacity
    return c


@pytest.mark.parametrize("name", LOGIT_SHAPES)
@pytest.mark.parametrize("quantize", [None, 0.25])
def test_topk_from_logits_bit_exact(name, quantize):
    s = SHAPES[name]
    T = s.T
    cfg = _cfg(s, T)
    z = _logits(T, s.E, seed=11, quantize=quantize)
    out = moe.topk_from_logits(cfg, z.to(DEV))
    torch.cuda.synchronize()
    ref = O.route(z.double().numpy(), s.k, s.gate, s.renormalize, s.rsf, None)
    np.testing.assert_array_equal(np_i(out["topk_idx"]), ref["topk_idx"])
    np.testing.assert_allclose(np_f(out["topk_w"]), ref["topk_w"], rtol=2e-6, atol=2e-7)
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], rtol=1e-4, atol=1e-6)


@pytest.mark.parametrize("gate,rsf,golden_key", [("softmax", 1.0, "softmax"),
                                                 ("sigmoid", 2.5, "sigmoid")])
def test_worked_example_on_gpu(golden, gate, rsf, golden_key):
    g = golden("moe10_gating_worked_example.json")
    cfg = moe.make_config(1, 64, 4, 2, 128, gate=gate, renormalize=True, rsf=rsf,
                          act_dtype="fp32")
    z = torch.tensor([g["logits"]], dtype=torch.float32, device=DEV)
    out = moe.topk_from_logits(cfg, z)
    torch.cuda.synchronize()
    assert out["topk_idx"].cpu().tolist() == [g["chosen"]]
    want = g[golden_key]["scaled"] if gate == "sigmoid" else g[golden_key]["renormalized"]
    np.testing.assert_allclose(np_f(out["topk_w"])[0], want, atol=5e-4)
    np.testing.assert_allclose(np_f(out["mean_prob"]), g[golden_key]["scores"], atol=5e-4)


def _dispatch_compare(cfg, idx_np, E, capacity):
    out = moe.dispatch(cfg, torch.from_numpy(idx_np.astype(np.int32)).to(DEV))
    torch.cuda.synchronize()
    ref = O.dispatch(idx_np, E, capacity)
    np.testing.assert_array_equal(np_i(out["counts"]), ref["counts"])
    np.testing.assert_array_equal(np_i(out["drops"]), ref["drops"])
    np.testing.assert_array_equal(np_i(out["offsets"]), ref["offsets"])
    n = int(ref["offsets"][-1])
    np.testing.assert_array_equal(np_i(out["perm"])[:n], ref["perm"][:n])
    A = idx_np.size
    np.testing.assert_array_equal(np_i(out["drop_mask"])[:A], ref["drop_mask"])
    return ref


@pytest.mark.parametrize("name", LOGIT_SHAPES)
def test_dispatch_bit_exact(name):
    s = SHAPES[name]
    z = _logits(s.T, s.E, seed=12).double().numpy()
    if s.zipf_s is not None:
        z = z - s.zipf_s * np.log(np.arange(s.E) + 1.0)
    idx = O.topk_experts(z, s.k)
    C = oracle_capacity(s)
    cfg = _cfg(s, s.T)
    ref = _dispatch_compare(cfg, idx, s.E, C)
    if s.capacity_factor is not None:
        assert ref["drops"].sum() > 0    # the skewed layer really overflows


@pytest.mark.parametrize("T,E,k,cap", [(1, 4, 2, -1), (5, 3, 3, 1), (4097, 8, 2, 900),
                                       (9000, 256, 8, 200), (7, 16, 4, 0), (20000, 64, 1, 100),
                                       (33, 1, 1, 5)])
def test_dispatch_edge_cases(T, E, k, cap):
    rng = np.random.default_rng(T + E)
    z = rng.normal(size=(T, E)) + np.linspace(2.0, 0.0, E)
    idx = O.topk_experts(z, k) if E * T < 2_000_000 else np.argsort(-z, axis=1, kind="stable")[:, :k]
    cfg = moe.make_config(T, 64, E, k, 128, act_dtype="bf16", capacity=cap)
    _dispatch_compare(cfg, idx, E, None if cap < 0 else cap)


def test_dispatch_reports_bad_expert_index():
    cfg = moe.make_config(8, 64, 4, 1, 128, act_dtype="bf16")
    ws = moe.Workspace(cfg)
    idx = torch.tensor([[0], [1], [7], [2], [3], [0], [1], [2]], dtype=torch.int32, device=DEV)
    moe.dispatch(cfg, idx, ws)
    assert moe.moe_get_error(ws) == moe._binding.MOE_ERR_DEVICE
    assert moe.moe_get_error(ws) == 0     # the status word is cleared by reading it


@pytest.mark.parametrize("name", LOGIT_SHAPES)
def test_router_end_to_end(name):
    s = SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=0, with_experts=False)
    cfg = _cfg(s, s.T)
    out = moe.route(cfg, inp["x"], inp["w_router"], inp["router_bias"])
    torch.cuda.synchronize()
    z64 = O.router_logits(to_f64(inp["x"]), to_f64(inp["w_router"]), to_f64(inp["router_bias"]))
    # logits: fp32 accumulation of bf16 products
    scale = np.sqrt(np.mean(z64 ** 2))
    np.testing.assert_allclose(np_f(out["logits"]), z64, atol=1e-4 * scale * np.sqrt(s.d / 128))
    ref = O.route(z64, s.k, s.gate, s.renormalize, s.rsf, None)
    margins = score_margins(ref["scores"], ref["topk_idx"])
    clear = margins > MARGIN
    gi = np_i(out["topk_idx"])
    # the margin fixes the chosen set; the order inside it is fixed where
    # consecutive chosen scores are separated by the margin as well
    sets = same_sets(gi, ref["topk_idx"])
    assert np.all(sets[clear])
    ordered = clear & order_separated(ref["scores"], ref["topk_idx"], MARGIN)
    assert np.array_equal(gi[ordered], ref["topk_idx"][ordered])
    same = np.all(gi == ref["topk_idx"], axis=1)
    assert same.mean() > 0.9
    np.testing.assert_allclose(np_f(out["topk_w"])[same], ref["topk_w"][same], atol=WEIGHT_ABS)
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], atol=1e-4)
