"""GPU parity of expert-choice routing (the amazingdata.cn article on MoE
routing, paragraph on expert choice: each expert takes a fixed number of the
tokens it scores highest; a token may be taken by no expert).

Fed the same fp32 logits, each expert's chosen tokens must equal the
oracle's whenever its C-th and (C+1)-th largest scores are separated by
more than SCORE_MARGIN (the kernel ranks fp32 scores; exact ties go to the
lower token on both sides, which quantised sigmoid logits exercise bit for
bit).  The layer output has the tolerances of the token-choice layer.
"""

import numpy as np
import pytest
import torch

import top_routing_expert_gate_b300 as moe
from oracle import moe_oracle as O
from workloads import SHAPES, MoEShape, make_inputs
from workloads.generate import to_f64

from gpu_util import assert_layer_close, layer_experts, layer_shared, np_f, np_i

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCORE_MARGIN = 1e-6


def _margin_ok(scores, C):
    """Per expert: the C-th / (C+1)-th score gap exceeds the margin."""
    T, E = scores.shape
    ok = np.ones(E, dtype=bool)
    if C == 0 or C >= T:
        return ok
    srt = -np.sort(-scores, axis=0)
    return (srt[C - 1] - srt[C]) > SCORE_MARGIN


CASES = [
    # T, E, k, capacity, gate, quantize
    (16384, 64, 1, -1, "softmax", None),
    (4096, 8, 2, -1, "sigmoid", None),
    (1000, 16, 2, -1, "softmax", None),
    (777, 12, 3, 100, "sigmoid", None),
    (300, 4, 1, 300, "softmax", None),       # C = T: every expert takes every token
    (50, 8, 1, 0, "sigmoid", None),          # C = 0
    (2048, 32, 4, -1, "sigmoid", 0.25),      # many exact score ties
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_E{c[1]}_k{c[2]}_C{c[3]}_{c[4]}" +
                                             ("_q" if c[5] else "") for c in CASES])
def test_expert_choice_from_logits(case):
    T, E, k, cap, gate, quant = case
    g = torch.Generator().manual_seed(T + E)
    z = torch.randn((T, E), generator=g, dtype=torch.float32)
    if quant:
        z = torch.round(z / quant) * quant
    cfg = moe.make_config(T, 64, E, k, 128, gate=gate, renormalize=False, capacity=cap,
                          act_dtype="fp32", routing="expert")
    C = moe.moe_expert_choice_capacity(cfg)
    assert C == O.expert_choice_capacity(T, E, k, None if cap < 0 else cap)
    out = moe.expert_choice_from_logits(cfg, z.to(DEV))
    torch.cuda.synchronize()
    scores = O.gate_scores(z.double().numpy(), gate)
    ref = O.expert_choice(scores, C)
    if C == 0:
        return
    toks = np_i(out["tokens"])
    # always: ascending, distinct, in range
    assert np.all(toks[:, 1:] > toks[:, :-1]) and toks.min() >= 0 and toks.max() < T
    ok = _margin_ok(scores, C) if not (quant and gate == "sigmoid") else np.ones(E, bool)
    assert ok.mean() > 0.9
    np.testing.assert_array_equal(toks[ok], ref["tokens"][ok])
    np.testing.assert_allclose(np_f(out["weights"])[ok], ref["weights"][ok], rtol=2e-6,
                               atol=1e-7)
    np.testing.assert_allclose(np_f(out["mean_prob"]), O.mean_router_prob(scores), rtol=1e-4,
                               atol=1e-6)


def _ec_shape(**kw):
    base = dict(name="ec", T=600, d=256, E=8, k=2, F=256, F_s=0, gate="softmax",
                renormalize=False, rsf=1.0, capacity_factor=None, zipf_s=None, dtype="bf16",
                routing="expert")
    base.update(kw)
    return MoEShape(**base)


EC_LAYERS = {
    "softmax": _ec_shape(),
    "sigmoid_shared": _ec_shape(T=333, d=192, E=16, k=4, F=384, F_s=256, gate="sigmoid"),
    "fp32": _ec_shape(T=77, d=64, E=5, k=3, F=96, F_s=32, dtype="fp32"),
    "ragged_ntail": _ec_shape(T=1000, d=320, E=4, k=2, F=256, F_s=128),
    "fp8_weights": _ec_shape(T=400, d=256, E=8, k=2, F=256, weight_format="fp8"),
}


def _near_threshold(scores, C, rel=2e-3):
    """Tokens with a score within rel (relative) of its expert's C-th largest
    score: with bf16 inputs the fp32 scores can rank them either way."""
    if C == 0:
        return np.zeros(scores.shape[0], dtype=bool)
    thr = (-np.sort(-scores, axis=0))[C - 1]
    return np.any(np.abs(scores - thr[None, :]) <= rel * thr[None, :] + 1e-7, axis=1)


def _oracle_ec(s, inp, C, tokens=None):
    return O.moe_layer_expert_choice(to_f64(inp["x"]), to_f64(inp["w_router"]),
                                     layer_experts(inp), C, s.gate, shared=layer_shared(inp),
                                     tokens=tokens)


@pytest.mark.parametrize("layout", ["tokens_m", "weights_m"])
@pytest.mark.parametrize("name", list(EC_LAYERS))
def test_expert_choice_layer_all_tokens(name, layout, monkeypatch):
    monkeypatch.setenv("MOE_B300_EXPERT_LAYOUT", layout)
    s = EC_LAYERS[name]
    inp = make_inputs(s, device=DEV, seed=14)
    cfg = moe.config_from_shape(s)
    C = moe.moe_expert_choice_capacity(cfg)
    ws = moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert "topk_idx" not in out
    np.testing.assert_array_equal(np_i(out["counts"]), np.full(s.E, C))
    np.testing.assert_array_equal(np_i(out["drops"]), np.zeros(s.E))
    ref = _oracle_ec(s, inp, C)
    # tokens whose set of choosing experts could flip (a score within the
    # end-to-end rounding of its expert's C-th largest) are left out
    near = _near_threshold(ref["scores"], C)
    assert (~near).mean() > 0.8
    assert_layer_close(np_f(out["y"])[~near], ref["y"][~near], name)
    np.testing.assert_allclose(np_f(out["mean_prob"]), ref["mean_prob"], atol=1e-4)


def test_expert_choice_full_capacity_matches_token_choice_top_E():
    # C = T with softmax: every expert takes every token, which is token
    # choice over all E experts with renormalisation (the weights sum to 1)
    s = _ec_shape(T=256, E=4, k=4)
    inp = make_inputs(s, device=DEV, seed=15)
    cfg = moe.config_from_shape(s)
    cfg.capacity = s.T
    a = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp))
    tc = moe.config_from_shape(MoEShape(**{**s.__dict__, "routing": "token", "renormalize": True}))
    b = moe.layer_forward(tc, inp["x"], moe.LayerWeights.from_inputs(inp))
    torch.cuda.synchronize()
    ya, yb = np_f(a["y"]), np_f(b["y"])
    # the same products summed in a different order (expert order vs logit order)
    np.testing.assert_allclose(ya, yb, rtol=0, atol=2e-6 * np.sqrt(np.mean(yb ** 2)) * 10)


@pytest.mark.slow
def test_full_size_switch_expert_choice_sampled():
    s = SHAPES["switch_expert_choice"]
    inp = make_inputs(s, device=DEV, seed=0)
    cfg = moe.config_from_shape(s)
    C = moe.moe_expert_choice_capacity(cfg)
    assert C == 256
    ws = moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    scores = O.gate_scores(O.router_logits(to_f64(inp["x"]), to_f64(inp["w_router"])), s.gate)
    near = _near_threshold(scores, C)
    assert (~near).sum() >= 24
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(np.arange(s.T)[~near], 24, replace=False))
    ref = _oracle_ec(s, inp, C, tokens=pick)
    assert_layer_close(np_f(out["y"])[pick], ref["y"], "switch expert choice")
    assert ref["picked"].sum() == s.E * C
