"""GPU parity of the layer with E4M3 expert weights (one fp32 scale per
output channel; "10. 混合专家 MoE：总参数与激活参数", section "推理时":
DeepSeek-V3 ships FP8 weights).

The oracle decodes the stored codes from the E4M3 definition and multiplies
by the scales, in float64.  The kernel widens the codes to bf16 on chip (exact)
and applies the scale to each output's fp32 accumulator, so the tolerances are
those of the bf16 layer.  With power-of-two scales the E4M3 layer must equal,
bit for bit, the bf16 layer run on the decoded weights.
"""

import numpy as np
import pytest
import torch

import top_routing_expert_gate_b300 as moe
from oracle import moe_oracle as O
from workloads import SHAPES, MoEShape, make_inputs

from workloads.generate import to_f64

from gpu_util import (MARGIN, assert_capacity_layer_close, assert_layer_close,
                      assert_routing_bit_exact, check_tokens, library_routing, np_f, np_i,
                      oracle_layer, oracle_route, same_sets, score_margins)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _shape(**kw):
    base = dict(name="fp8", T=300, d=256, E=8, k=2, F=384, F_s=0, gate="softmax",
                renormalize=True, rsf=1.0, capacity_factor=None, zipf_s=None, dtype="bf16",
                weight_format="fp8")
    base.update(kw)
    return MoEShape(**base)


FP8_SHAPES = {
    "softmax": _shape(),
    "sigmoid_shared": _shape(T=257, d=192, E=16, k=4, F=256, F_s=384, gate="sigmoid", rsf=2.5),
    "multi_mtile_ntail": _shape(T=1000, d=320, E=4, k=2, F=256, F_s=128),
    "capacity": _shape(T=999, d=128, E=8, k=1, F=256, renormalize=False, capacity_factor=1.25,
                       zipf_s=1.2),
    # shapes for the weights-in-M kernel (d_model a multiple of 256): a few
    # rows per expert; several 64-token tiles per expert with a ragged last
    # one and a shared expert over 5 token tiles; capacity with drops
    "decode_shared": _shape(T=40, d=512, E=32, k=4, F=256, F_s=256, gate="sigmoid", rsf=2.5),
    "tm_multi_tile": _shape(T=300, d=256, E=4, k=2, F=384, F_s=128),
    "tm_capacity": _shape(T=700, d=256, E=8, k=2, F=256, capacity_factor=1.0, zipf_s=1.2),
}

# MOE_B300_FP8_LAYOUT: tokens in M (weights widened to bf16 in shared
# memory) or weights in M (widened into tensor memory) with token tiles of 32,
# 64 or 128 rows, whose operands are fp16 (tokens rescaled per row) or, with
# MOE_B300_FP8_TOKENS=bf16, bf16; shapes the weights-in-M kernel does not
# support fall back to tokens in M
FP8_LAYOUTS = ["tokens_m", "weights_tm32", "weights_tm", "weights_tm128", "weights_tm_bf16",
               "weights_tm32_bf16"]


def _set_fp8_layout(monkeypatch, layout):
    monkeypatch.setenv("MOE_B300_FP8_LAYOUT", layout.replace("_bf16", ""))
    if layout.endswith("_bf16"):
        monkeypatch.setenv("MOE_B300_FP8_TOKENS", "bf16")
    else:
        monkeypatch.delenv("MOE_B300_FP8_TOKENS", raising=False)


def _check_layer(s, inp, cfg, ws, out):
    """The layer against the oracle routed from the library's fp32 logits:
    routing and dispatch bit for bit, the output on every token (capacity
    layers included); then the end-to-end routing rule on margin-clear
    tokens."""
    lib = library_routing(cfg, inp, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(lib["topk_idx"], out["topk_idx"])
    ref = oracle_layer(s, inp, logits=np_f(lib["logits"]))
    assert_routing_bit_exact(lib, ref, s.T, s.k)
    if s.capacity_factor is None:
        assert_layer_close(np_f(out["y"]), ref["y"], s.name)
    else:
        assert ref["drops"].sum() > 0
        assert_capacity_layer_close(np_f(out["y"]), ref["y"], ref["drop_mask"], s.name)
    ref_b = oracle_route(s, O.router_logits(to_f64(inp["x"]), to_f64(inp["w_router"]),
                                            to_f64(inp["router_bias"])))
    same = same_sets(np_i(out["topk_idx"]), ref_b["topk_idx"])
    assert np.all(same[score_margins(ref_b["scores"], ref_b["topk_idx"]) > MARGIN])


@pytest.mark.parametrize("layout", FP8_LAYOUTS)
@pytest.mark.parametrize("name", list(FP8_SHAPES))
def test_fp8_layer_matches_oracle_all_tokens(name, layout, monkeypatch):
    _set_fp8_layout(monkeypatch, layout)
    s = FP8_SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=11)
    assert inp["w_gate"].dtype == torch.float8_e4m3fn
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    _check_layer(s, inp, cfg, ws, out)


def _every_code(shape_, gen):
    """Random E4M3 codes covering every finite code (0x7F / 0xFF excluded)."""
    finite = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    idx = torch.randint(0, len(finite), shape_, generator=gen)
    codes = finite[idx]
    flat = codes.view(-1)
    flat[: len(finite)] = finite            # each code at least once
    return codes.view(torch.float8_e4m3fn)


@pytest.mark.parametrize("layout", FP8_LAYOUTS)
def test_fp8_every_code_decodes_like_the_oracle(layout, monkeypatch):
    # weights made of all 254 finite codes (subnormals, 448, both signs) with
    # non-power-of-two scales; the layer must match the oracle's decoding
    _set_fp8_layout(monkeypatch, layout)
    s = _shape(T=200, d=256, E=2, k=2, F=256, gate="sigmoid", rsf=2.5)
    inp = make_inputs(s, device=DEV, seed=12)
    g = torch.Generator().manual_seed(3)
    for key, rows in (("w_gate", (2, 256, 256)), ("w_up", (2, 256, 256)), ("w_down", (2, 256, 256))):
        inp[key] = _every_code(rows, g).to(DEV)
        fan_in = 256
        inp[key + "_scale"] = (torch.rand(rows[:2], generator=g) * 0.5 + 0.5).mul(
            1.0 / (200.0 * np.sqrt(fan_in))).to(DEV)
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    _check_layer(s, inp, cfg, ws, out)


@pytest.mark.parametrize("layout", FP8_LAYOUTS)
@pytest.mark.parametrize("F_s", [0, 256])
def test_fp8_equals_bf16_on_decoded_weights_with_power_of_two_scales(F_s, layout, monkeypatch):
    # the bf16 layer runs with the same MMA orientation (weights in M for the
    # tensor-memory kernel), so the products and sums are the same
    _set_fp8_layout(monkeypatch, layout)
    monkeypatch.setenv("MOE_B300_EXPERT_LAYOUT", "tokens_m" if layout == "tokens_m" else "weights_m")
    s = _shape(T=515, d=256, E=8, k=2, F=256, F_s=F_s, gate="sigmoid", rsf=2.5)
    inp = make_inputs(s, device=DEV, seed=13)
    g = torch.Generator().manual_seed(4)
    keys = ["w_gate", "w_up", "w_down"] + (["ws_gate", "ws_up", "ws_down"] if F_s else [])
    bf = dict(inp)
    for key in keys:
        sc = inp[key + "_scale"]
        p2 = torch.exp2(torch.round(torch.log2(sc.float()))).to(DEV)   # nearest power of two
        inp[key + "_scale"] = p2
        dec = inp[key].float() * p2.unsqueeze(-1)                      # exact in bf16
        bf[key] = dec.to(torch.bfloat16)
        assert torch.equal(bf[key].float(), dec)
        bf[key + "_scale"] = None
    cfg8 = moe.config_from_shape(s)
    cfgb = moe.config_from_shape(MoEShape(**{**s.__dict__, "weight_format": "act"}))
    o8 = moe.layer_forward(cfg8, inp["x"], moe.LayerWeights.from_inputs(inp))
    ob = moe.layer_forward(cfgb, bf["x"], moe.LayerWeights.from_inputs(bf))
    torch.cuda.synchronize()
    assert torch.equal(o8["topk_idx"], ob["topk_idx"])
    assert torch.equal(o8["y"], ob["y"])


@pytest.mark.slow
@pytest.mark.parametrize("name,n_check", [("dsv3_decode_fp8", 64), ("dsv3_prefill_fp8", 320)])
def test_full_size_fp8_layer_sampled(name, n_check):
    # the benchmark's launch configuration; the decode batch is compared on
    # all 64 tokens, prefill on every expert's ragged-tail token plus random ones
    s = SHAPES[name]
    inp = make_inputs(s, device=DEV, seed=0)
    cfg = moe.config_from_shape(s)
    ws = moe.Workspace(cfg)
    out = moe.layer_forward(cfg, inp["x"], moe.LayerWeights.from_inputs(inp), ws=ws)
    lib = library_routing(cfg, inp, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(lib["topk_idx"], out["topk_idx"])
    ref = oracle_route(s, np_f(lib["logits"]))
    assert_routing_bit_exact(lib, ref, s.T, s.k)
    z = O.router_logits(to_f64(inp["x"]), to_f64(inp["w_router"]))
    ref_b = oracle_route(s, z)
    same = same_sets(np_i(out["topk_idx"]), ref_b["topk_idx"])
    assert np.all(same[score_margins(ref_b["scores"], ref_b["topk_idx"]) > MARGIN])
    pick = check_tokens(ref, s.T, s.k, n_check)
    assert len(pick) >= min(n_check, s.T)
    oref = oracle_layer(s, inp, tokens=pick, logits=np_f(lib["logits"]))
    assert_layer_close(np_f(out["y"])[pick], oref["y"], name)
