"""The C ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host before anything reaches the GPU.  No GPU is needed:
every call here either is host-only or fails validation before any launch."""

import ctypes
import os
import re

import pytest

import top_routing_expert_gate_b300 as moe
from top_routing_expert_gate_b300 import _binding as B
from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                src = f.read()
            names |= set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_symbol():
    lib = B.load_library()
    declared = _declared_symbols()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
    # and the binding declares a signature for each of them
    assert declared <= set(B.SIGNATURES)


def test_exported_symbols_in_dynamic_table():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, flags=re.M))
    assert _declared_symbols() <= exported


def test_version_and_status_strings():
    lib = B.load_library()
    assert moe.moe_version() >= 100
    for code in range(7):
        assert lib.moe_status_string(code).decode().startswith("MOE_")


@pytest.mark.parametrize("T,E,cf", [(8, 4, 1.0), (8, 4, 1.25), (8, 4, 2.5), (16384, 64, 1.25),
                                    (1000, 7, 1.1), (3, 5, 0.0), (0, 4, 1.0), (65536, 256, 1.3)])
def test_capacity_matches_oracle(T, E, cf):
    assert moe.moe_capacity(T, E, cf) == O.expert_capacity(T, E, cf)


def test_capacity_rejects_bad_args():
    assert moe.moe_capacity(-1, 4, 1.0) == -1
    assert moe.moe_capacity(8, 0, 1.0) == -1
    assert moe.moe_capacity(8, 4, -0.5) == -1
    assert moe.moe_capacity(8, 4, float("nan")) == -1


def _cfg(**kw):
    base = dict(T=64, d=128, E=4, k=2, F=256, F_s=0, gate="softmax", renormalize=True, rsf=1.0,
                capacity=-1, act_dtype="fp32", out_dtype="fp32")
    base.update(kw)
    return moe.make_config(**base)


def _ws_size(cfg):
    n = ctypes.c_size_t(0)
    return B.load_library().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), n.value


def test_workspace_size_grows_with_shape():
    s1, n1 = _ws_size(_cfg())
    s2, n2 = _ws_size(_cfg(T=128))
    assert s1 == 0 and s2 == 0 and n2 > n1 > 0


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(k=5), B.MOE_ERR_INVALID_ARG),          # k > E
    (dict(k=0), B.MOE_ERR_INVALID_ARG),
    (dict(E=0), B.MOE_ERR_INVALID_ARG),
    (dict(E=300, k=2), B.MOE_ERR_UNSUPPORTED),   # > 256 experts
    (dict(E=64, k=33), B.MOE_ERR_UNSUPPORTED),   # > 32 choices
    (dict(d=130), B.MOE_ERR_UNSUPPORTED),        # d not a multiple of 4
    (dict(act_dtype="bf16", d=96), B.MOE_ERR_UNSUPPORTED),    # bf16 needs d % 64
    (dict(act_dtype="bf16", F=200), B.MOE_ERR_UNSUPPORTED),   # bf16 needs F % 128
    (dict(F=0), B.MOE_ERR_INVALID_ARG),
])
def test_config_validation(kw, code):
    assert _ws_size(_cfg(**kw))[0] == code


def test_bad_gate_and_dtype_enums():
    c = _cfg()
    c.gate = 7
    assert _ws_size(c)[0] == B.MOE_ERR_INVALID_ARG
    c = _cfg()
    c.act_dtype = 9
    assert _ws_size(c)[0] == B.MOE_ERR_INVALID_ARG
    c = _cfg()
    c.renormalize = 2
    assert _ws_size(c)[0] == B.MOE_ERR_INVALID_ARG


def test_entry_points_reject_missing_workspace_and_pointers():
    lib = B.load_library()
    cfg = _cfg()
    _, need = _ws_size(cfg)
    fake = 0x10000   # never dereferenced: validation fails before any launch
    # workspace too small / misaligned / null
    assert lib.moe_topk_from_logits(ctypes.byref(cfg), fake, None, fake, fake, None, fake, need - 1,
                                    None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_topk_from_logits(ctypes.byref(cfg), fake, None, fake, fake, None, fake + 16, need,
                                    None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_topk_from_logits(ctypes.byref(cfg), fake, None, fake, fake, None, None, need,
                                    None) == B.MOE_ERR_WORKSPACE
    # null required pointer
    assert lib.moe_topk_from_logits(ctypes.byref(cfg), None, None, fake, fake, None, fake, need,
                                    None) == B.MOE_ERR_INVALID_ARG
    # misaligned logits
    assert lib.moe_topk_from_logits(ctypes.byref(cfg), fake + 4, None, fake, fake, None, fake, need,
                                    None) == B.MOE_ERR_INVALID_ARG
    # dispatch: null counts
    assert lib.moe_dispatch(ctypes.byref(cfg), fake, None, fake, fake, fake, fake, fake, need,
                            None) == B.MOE_ERR_INVALID_ARG
    # layer: shared weights given although d_ff_shared == 0
    assert lib.moe_layer_forward(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake, fake,
                                 fake, fake, None, None, fake, None, None, None, None, None, fake,
                                 need, None) == B.MOE_ERR_INVALID_ARG
    # layer: only some shared weights
    cs = _cfg(F_s=128)
    _, need_s = _ws_size(cs)
    assert lib.moe_layer_forward(ctypes.byref(cs), fake, fake, None, None, fake, fake, fake, fake,
                                 None, fake, None, None, fake, None, None, None, None, None, fake,
                                 need_s, None) == B.MOE_ERR_INVALID_ARG
    # layer: a shared-expert gate without a shared expert
    assert lib.moe_layer_forward(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake,
                                 None, None, None, fake, None, fake, None, None, None, None, None,
                                 fake, need, None) == B.MOE_ERR_INVALID_ARG
    # E4M3 weights: scales required, and only with bf16 activations
    c8 = _cfg(act_dtype="bf16", weight_format="fp8")
    _, need8 = _ws_size(c8)
    assert lib.moe_layer_forward(ctypes.byref(c8), fake, fake, None, None, fake, fake, fake,
                                 None, None, None, None, None, fake, None, None, None, None, None,
                                 fake, need8, None) == B.MOE_ERR_INVALID_ARG
    sc = B.MoEWeightScales(fake, fake, fake + 4, None, None, None)   # misaligned down scales
    assert lib.moe_layer_forward(ctypes.byref(c8), fake, fake, None, None, fake, fake, fake,
                                 None, None, None, None, ctypes.byref(sc), fake, None, None, None,
                                 None, None, fake, need8, None) == B.MOE_ERR_INVALID_ARG
    sc_ok = B.MoEWeightScales(fake, fake, fake, None, None, None)
    assert lib.moe_layer_forward(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake,
                                 None, None, None, None, ctypes.byref(sc_ok), fake, None, None,
                                 None, None, None, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert _ws_size(_cfg(act_dtype="fp32", weight_format="fp8"))[0] == B.MOE_ERR_UNSUPPORTED
    # host-buffer call: null host x or host y
    assert lib.moe_layer_forward_host(ctypes.byref(cfg), None, fake, fake, None, None, fake, fake,
                                      fake, None, None, None, None, None, fake, fake, None, None,
                                      None, None, None, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_host(ctypes.byref(cfg), fake, fake, fake, None, None, fake, fake,
                                      fake, None, None, None, None, None, fake, None, None, None,
                                      None, None, None, fake, need, None) == B.MOE_ERR_INVALID_ARG
    # null config
    assert lib.moe_layer_forward(None, fake, fake, None, None, fake, fake, fake, None, None, None,
                                 None, None, fake, None, None, None, None, None, fake, need,
                                 None) == B.MOE_ERR_INVALID_ARG
    # balance loss / shared gate: null outputs
    assert lib.moe_balance_loss(ctypes.byref(cfg), fake, None, fake, 0.01, None,
                                None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_shared_gate_weights(ctypes.byref(cfg), fake, None, fake,
                                       None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_get_error(None, None) == B.MOE_ERR_WORKSPACE
    # misaligned selection bias
    assert lib.moe_topk_from_logits(ctypes.byref(cfg), fake, fake + 4, fake, fake, None, fake,
                                    need, None) == B.MOE_ERR_INVALID_ARG
    # score-bias step: null counts / bias, non-finite gamma
    assert lib.moe_update_score_bias(ctypes.byref(cfg), None, None, 0.001, fake,
                                     None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_update_score_bias(ctypes.byref(cfg), fake, None, 0.001, None,
                                     None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_update_score_bias(ctypes.byref(cfg), fake, None, float("nan"), fake,
                                     None) == B.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("E,k,n_group,topk_group,want", [
    (256, 8, 8, 4, B.MOE_OK),               # DeepSeek-V3: 8 groups of 32, keep 4
    (16, 2, 0, 0, B.MOE_OK),                # no groups
    (16, 2, 1, 0, B.MOE_OK),                # one group = no groups
    (16, 2, 3, 1, B.MOE_ERR_INVALID_ARG),   # 3 does not divide 16
    (16, 2, 16, 4, B.MOE_ERR_INVALID_ARG),  # groups of one expert
    (16, 2, 4, 0, B.MOE_ERR_INVALID_ARG),   # no group kept
    (16, 2, 4, 5, B.MOE_ERR_INVALID_ARG),   # more groups kept than exist
    (16, 9, 4, 2, B.MOE_ERR_INVALID_ARG),   # k larger than the kept experts (8)
    (128, 2, 64, 4, B.MOE_ERR_UNSUPPORTED), # more than 32 groups
    (16, 2, -1, 0, B.MOE_ERR_INVALID_ARG),
])
def test_group_fields_validated(E, k, n_group, topk_group, want):
    c = _cfg(E=E, k=k)
    c.n_group = n_group
    c.topk_group = topk_group
    assert _ws_size(c)[0] == want


def test_expert_choice_config_and_capacity():
    lib = B.load_library()
    c = _cfg(T=10, E=4, k=2, routing="expert")
    assert lib.moe_expert_choice_capacity(ctypes.byref(c)) == 5        # ceil(10 * 2 / 4)
    c.capacity = 3
    assert lib.moe_expert_choice_capacity(ctypes.byref(c)) == 3
    c.capacity = 99
    assert lib.moe_expert_choice_capacity(ctypes.byref(c)) == 10       # at most T
    big = _cfg(T=40000, E=4, k=2, routing="expert")
    assert _ws_size(big)[0] == B.MOE_ERR_UNSUPPORTED
    grouped = _cfg(E=8, k=2, routing="expert")
    grouped.n_group, grouped.topk_group = 4, 2
    assert _ws_size(grouped)[0] == B.MOE_ERR_INVALID_ARG
    bad = _cfg()
    bad.routing = 5
    assert _ws_size(bad)[0] == B.MOE_ERR_INVALID_ARG
    # token-choice entry points refuse an expert-choice configuration
    ec = _cfg(routing="expert")
    _, need = _ws_size(ec)
    fake = 0x10000
    assert lib.moe_topk_from_logits(ctypes.byref(ec), fake, None, fake, fake, None, fake, need,
                                    None) == B.MOE_ERR_INVALID_ARG
    # expert-choice layer forward rejects per-token top-k outputs
    assert lib.moe_layer_forward(ctypes.byref(ec), fake, fake, None, None, fake, fake, fake,
                                 None, None, None, None, None, fake, fake, None, None, None, None,
                                 fake, need, None) == B.MOE_ERR_INVALID_ARG


def test_config_from_shape_capacity():
    from workloads import SHAPES
    c = moe.config_from_shape(SHAPES["switch"])
    assert c.capacity == 320 and c.top_k == 1 and c.renormalize == 0
    c = moe.config_from_shape(SHAPES["dsv3_prefill"])
    assert c.capacity == -1 and abs(c.routed_scaling_factor - 2.5) < 1e-7 and c.gate == 1


def test_no_workspace_dispatch_applies_the_dispatch_config_rules():
    # moe_dispatch_no_workspace validates the configuration as moe_dispatch
    # does (and refuses expert-choice routing) before any CUDA call
    lib = B.load_library()
    fake = 0x10000   # never dereferenced: validation fails first

    def call(c):
        return lib.moe_dispatch_no_workspace(ctypes.byref(c), fake, fake, fake, fake, fake, fake,
                                             None)

    assert call(_cfg(routing="expert")) == B.MOE_ERR_INVALID_ARG
    c = _cfg()
    c.gate = 7
    assert call(c) == B.MOE_ERR_INVALID_ARG
    c = _cfg()
    c.d_ff = 0
    assert call(c) == B.MOE_ERR_INVALID_ARG
    c = _cfg()
    c.top_k = c.n_experts + 1
    assert call(c) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch_no_workspace(None, fake, fake, fake, fake, fake, fake,
                                         None) == B.MOE_ERR_INVALID_ARG
    # misaligned output pointer
    assert lib.moe_dispatch_no_workspace(ctypes.byref(_cfg()), fake, fake + 4, fake, fake, fake,
                                         fake, None) == B.MOE_ERR_INVALID_ARG
