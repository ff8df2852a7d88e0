"""The seeded input generator: determinism, shapes and the stated recipe."""

import math

import numpy as np
import torch

from workloads import SHAPES, make_inputs, tensor_seed
from workloads.generate import ExpertWeights, to_f64


def test_seeds_are_stable_and_distinct():
    assert tensor_seed(0, "x") == tensor_seed(0, "x")
    assert tensor_seed(0, "x") != tensor_seed(1, "x")
    assert tensor_seed(0, "w_gate.0") != tensor_seed(0, "w_gate.1")


def test_tiny_inputs_deterministic_and_shaped():
    s = SHAPES["tiny"]
    a = make_inputs(s, seed=0)
    b = make_inputs(s, seed=0)
    for k in ("x", "w_router", "w_gate", "w_up", "w_down"):
        assert torch.equal(a[k], b[k])
    assert a["x"].shape == (64, 128) and a["x"].dtype == torch.float32
    assert a["w_gate"].shape == (4, 256, 128)
    assert a["w_down"].shape == (4, 128, 256)
    assert a["router_bias"] is None and a["ws_gate"] is None


def test_recipe_scales():
    s = SHAPES["tiny"].with_tokens(4096)
    a = make_inputs(s, seed=3)
    assert abs(a["x"].std().item() - 1.0) < 0.02
    assert abs(a["w_router"].std().item() * math.sqrt(s.d) - 1.0) < 0.05
    assert abs(a["w_down"].std().item() * math.sqrt(s.F) - 1.0) < 0.02


def test_zipf_bias_and_expert_view():
    s = SHAPES["switch"]
    small = type(s)(**{**s.__dict__, "T": 8, "d": 16, "F": 32})
    a = make_inputs(small, seed=0)
    b = a["router_bias"].double().numpy()
    assert b[0] == 0.0
    np.testing.assert_allclose(b, -1.2 * np.log(np.arange(64) + 1.0), rtol=1e-6)
    assert a["x"].dtype == torch.bfloat16
    ew = ExpertWeights(a["w_gate"], a["w_up"], a["w_down"])
    wg, wu, wd = ew[5]
    assert wg.dtype == np.float64 and wg.shape == (32, 16) and wd.shape == (16, 32)
    np.testing.assert_array_equal(wg, to_f64(a["w_gate"][5]))
