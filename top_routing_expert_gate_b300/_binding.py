"""ctypes declarations of libmoe_b300.so (include/moe_b300.h), nothing more.

Loading fails loudly when the shared library has not been built: there is no
fallback implementation of any step.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_size_t, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE = 6

MOE_NUM_STAGES = 7
STAGE_NAMES = ("router", "topk", "dispatch", "gather", "gate_up", "down", "combine")

MOE_GATE_SOFTMAX = 0
MOE_GATE_SIGMOID = 1
MOE_BF16 = 0
MOE_FP32 = 1
MOE_WEIGHTS_ACT = 0
MOE_WEIGHTS_FP8_E4M3 = 1
MOE_ROUTE_TOKEN_CHOICE = 0
MOE_ROUTE_EXPERT_CHOICE = 1


class MoEConfig(ctypes.Structure):
    """Mirror of moe_config_t."""
    _fields_ = [
        ("T", c_int32),
        ("d_model", c_int32),
        ("n_experts", c_int32),
        ("top_k", c_int32),
        ("d_ff", c_int32),
        ("d_ff_shared", c_int32),
        ("gate", c_int32),
        ("renormalize", c_int32),
        ("routed_scaling_factor", c_float),
        ("capacity", c_int32),
        ("act_dtype", c_int32),
        ("out_dtype", c_int32),
        ("n_group", c_int32),
        ("topk_group", c_int32),
        ("weight_format", c_int32),
        ("routing", c_int32),
    ]

    def __repr__(self):
        return "MoEConfig(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class MoEWeightScales(ctypes.Structure):
    """Mirror of moe_weight_scales_t (device pointers)."""
    _fields_ = [
        ("gate_scale", c_void_p),
        ("up_scale", c_void_p),
        ("down_scale", c_void_p),
        ("shared_gate_scale", c_void_p),
        ("shared_up_scale", c_void_p),
        ("shared_down_scale", c_void_p),
    ]


CFG = POINTER(MoEConfig)
SCALES = POINTER(MoEWeightScales)
_I32P = c_void_p   # device pointers are passed as plain addresses

# name -> (restype, argtypes); every function of include/moe_b300.h
SIGNATURES = {
    "moe_version": (c_int32, []),
    "moe_status_string": (c_char_p, [c_int32]),
    "moe_capacity": (c_int32, [c_int32, c_int32, c_double]),
    "moe_workspace_size": (c_int32, [CFG, POINTER(c_size_t)]),
    "moe_workspace_init": (c_int32, [CFG, c_void_p, c_size_t, c_void_p]),
    "moe_router_topk": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_topk_from_logits": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_size_t, c_void_p]),
    "moe_update_score_bias": (c_int32, [CFG, c_void_p, c_void_p, c_float, c_void_p, c_void_p]),
    "moe_expert_choice_capacity": (c_int32, [CFG]),
    "moe_expert_choice_from_logits": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p,
                                                c_void_p, c_size_t, c_void_p]),
    "moe_dispatch": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_no_workspace": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_void_p, c_void_p]),
    "moe_grouped_swiglu": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, SCALES, c_void_p,
                                     c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_combine": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_shared_gate_weights": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_balance_loss": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_float, c_void_p,
                                   c_void_p]),
    "moe_layer_forward": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, SCALES, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_layer_forward_host": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, SCALES, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_size_t, c_void_p]),
    "moe_layer_forward_profiled": (c_int32, [CFG, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, SCALES, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_size_t, c_void_p, c_void_p, c_void_p]),
    "moe_get_error": (c_int32, [c_void_p, c_void_p]),
    "moe_selftest_bounded_wait": (c_int32, [c_void_p, c_size_t, ctypes.c_uint64, c_void_p]),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library once; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: the CUDA library must be built first "
            "(python -m top_routing_expert_gate_b300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = load_library()
        self.code = code
        super().__init__(f"{where}: {lib.moe_status_string(code).decode()}")


def check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoEError(code, where)
