"""Torch-facing binding of the C ABI: argument marshalling only.

Every function named ``moe_*`` here calls the C function of the same name in
libmoe_b300.so with the tensors' device addresses and the current CUDA
stream.  torch supplies device memory and streams; every step of the layer
runs in the library's own kernels.  The helpers ``route``, ``dispatch`` and
``layer_forward`` only allocate outputs and call those functions.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Dict, Optional

import torch

from . import _binding as B
from ._binding import MoEConfig, check, load_library

_DT = {"bf16": B.MOE_BF16, "fp32": B.MOE_FP32}
_TORCH_DT = {B.MOE_BF16: torch.bfloat16, B.MOE_FP32: torch.float32}


_WF = {"act": B.MOE_WEIGHTS_ACT, "fp8": B.MOE_WEIGHTS_FP8_E4M3}
_RT = {"token": B.MOE_ROUTE_TOKEN_CHOICE, "expert": B.MOE_ROUTE_EXPERT_CHOICE}


def make_config(T: int, d: int, E: int, k: int, F: int, F_s: int = 0, gate: str = "softmax",
                renormalize: bool = True, rsf: float = 1.0, capacity: int = -1,
                act_dtype: str = "bf16", out_dtype: str = "fp32", n_group: int = 0,
                topk_group: int = 0, weight_format: str = "act",
                routing: str = "token") -> MoEConfig:
    return MoEConfig(T=T, d_model=d, n_experts=E, top_k=k, d_ff=F, d_ff_shared=F_s,
                     gate=B.MOE_GATE_SOFTMAX if gate == "softmax" else B.MOE_GATE_SIGMOID,
                     renormalize=1 if renormalize else 0, routed_scaling_factor=float(rsf),
                     capacity=int(capacity), act_dtype=_DT[act_dtype], out_dtype=_DT[out_dtype],
                     n_group=int(n_group), topk_group=int(topk_group),
                     weight_format=_WF[weight_format], routing=_RT[routing])


def config_from_shape(shape, out_dtype: str = "fp32", T: Optional[int] = None) -> MoEConfig:
    """moe_config_t for a workloads.MoEShape (capacity from its factor)."""
    T = shape.T if T is None else T
    cap = -1
    if shape.capacity_factor is not None:
        cap = moe_capacity(T, shape.E, shape.capacity_factor)
    return make_config(T, shape.d, shape.E, shape.k, shape.F, shape.F_s, shape.gate,
                       shape.renormalize, shape.rsf, cap, shape.dtype, out_dtype,
                       getattr(shape, "n_group", 0), getattr(shape, "topk_group", 0),
                       getattr(shape, "weight_format", "act"), getattr(shape, "routing", "token"))


def act_dtype(cfg: MoEConfig) -> torch.dtype:
    return _TORCH_DT[cfg.act_dtype]


def out_dtype(cfg: MoEConfig) -> torch.dtype:
    return _TORCH_DT[cfg.out_dtype]


def _ptr(t: Optional[torch.Tensor], name: str = "tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------------------
# C ABI, one wrapper per entry point
# ---------------------------------------------------------------------------

def moe_version() -> int:
    return load_library().moe_version()


def moe_capacity(T: int, E: int, capacity_factor: float) -> int:
    return load_library().moe_capacity(T, E, float(capacity_factor))


def moe_workspace_size(cfg: MoEConfig) -> int:
    n = ctypes.c_size_t(0)
    check(load_library().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
          "moe_workspace_size")
    return n.value


class Workspace:
    """Device workspace for one configuration (torch-allocated, zero status)."""

    def __init__(self, cfg: MoEConfig, device="cuda"):
        self.nbytes = moe_workspace_size(cfg)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        self.ptr = (base + 255) // 256 * 256
        check(load_library().moe_workspace_init(ctypes.byref(cfg), self.ptr, self.nbytes,
                                                _stream(None)), "moe_workspace_init")


def moe_router_topk(cfg, x, w_router, router_bias, score_bias, logits_out, topk_idx, topk_w,
                    mean_prob, ws: Workspace, stream=None) -> None:
    check(load_library().moe_router_topk(
        ctypes.byref(cfg), _ptr(x, "x"), _ptr(w_router, "w_router"), _ptr(router_bias),
        _ptr(score_bias), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(mean_prob),
        ws.ptr, ws.nbytes, _stream(stream)), "moe_router_topk")


def moe_topk_from_logits(cfg, logits, score_bias, topk_idx, topk_w, mean_prob, ws: Workspace,
                         stream=None) -> None:
    check(load_library().moe_topk_from_logits(
        ctypes.byref(cfg), _ptr(logits, "logits"), _ptr(score_bias), _ptr(topk_idx),
        _ptr(topk_w), _ptr(mean_prob), ws.ptr, ws.nbytes, _stream(stream)),
        "moe_topk_from_logits")


def moe_expert_choice_capacity(cfg) -> int:
    return load_library().moe_expert_choice_capacity(ctypes.byref(cfg))


def moe_expert_choice_from_logits(cfg, logits, tokens, weights, mean_prob, ws: Workspace,
                                  stream=None) -> None:
    check(load_library().moe_expert_choice_from_logits(
        ctypes.byref(cfg), _ptr(logits, "logits"), _ptr(tokens), _ptr(weights), _ptr(mean_prob),
        ws.ptr, ws.nbytes, _stream(stream)), "moe_expert_choice_from_logits")


def expert_choice_from_logits(cfg, logits, ws: Optional[Workspace] = None):
    dev = logits.device
    ws = ws or Workspace(cfg, dev)
    C, E = moe_expert_choice_capacity(cfg), cfg.n_experts
    out = {"tokens": torch.empty((E, C), dtype=torch.int32, device=dev),
           "weights": torch.empty((E, C), dtype=torch.float32, device=dev),
           "mean_prob": _f32(E, dev)}
    moe_expert_choice_from_logits(cfg, logits, out["tokens"] if C else None,
                                  out["weights"] if C else None, out["mean_prob"], ws)
    return out


def moe_update_score_bias(cfg, counts, drops, gamma: float, score_bias, stream=None) -> None:
    check(load_library().moe_update_score_bias(
        ctypes.byref(cfg), _ptr(counts, "counts"), _ptr(drops), float(gamma),
        _ptr(score_bias, "score_bias"), _stream(stream)), "moe_update_score_bias")


def moe_dispatch(cfg, topk_idx, counts, drops, offsets, perm, drop_mask, ws: Workspace,
                 stream=None) -> None:
    check(load_library().moe_dispatch(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(drops), _ptr(offsets),
        _ptr(perm), _ptr(drop_mask), ws.ptr, ws.nbytes, _stream(stream)), "moe_dispatch")


@dataclass
class WeightScales:
    """Per-output-channel fp32 scales of E4M3 expert weights (moe_weight_scales_t)."""
    gate: torch.Tensor                 # [E, F]
    up: torch.Tensor                   # [E, F]
    down: torch.Tensor                 # [E, d]
    shared_gate: Optional[torch.Tensor] = None   # [F_s]
    shared_up: Optional[torch.Tensor] = None     # [F_s]
    shared_down: Optional[torch.Tensor] = None   # [d]

    def as_c(self) -> B.MoEWeightScales:
        return B.MoEWeightScales(_ptr(self.gate, "gate scale"), _ptr(self.up, "up scale"),
                                 _ptr(self.down, "down scale"), _ptr(self.shared_gate),
                                 _ptr(self.shared_up), _ptr(self.shared_down))

    @classmethod
    def from_inputs(cls, inputs) -> Optional["WeightScales"]:
        if inputs.get("w_gate_scale") is None:
            return None
        return cls(inputs["w_gate_scale"], inputs["w_up_scale"], inputs["w_down_scale"],
                   inputs.get("ws_gate_scale"), inputs.get("ws_up_scale"),
                   inputs.get("ws_down_scale"))


def _scales_ref(scales: Optional[WeightScales]):
    return None if scales is None else ctypes.byref(scales.as_c())


def moe_grouped_swiglu(cfg, x, perm, offsets, w_gate, w_up, w_down, ws_gate, ws_up, ws_down,
                       y_perm, y_shared, ws: Workspace, stream=None,
                       scales: Optional[WeightScales] = None) -> None:
    check(load_library().moe_grouped_swiglu(
        ctypes.byref(cfg), _ptr(x), _ptr(perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), _scales_ref(scales),
        _ptr(y_perm), _ptr(y_shared), ws.ptr, ws.nbytes, _stream(stream)),
        "moe_grouped_swiglu")


def moe_combine(cfg, y_perm, topk_w, offsets, perm, drop_mask, y_shared, shared_weight, y,
                ws: Workspace, stream=None) -> None:
    check(load_library().moe_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(topk_w), _ptr(offsets), _ptr(perm),
        _ptr(drop_mask), _ptr(y_shared), _ptr(shared_weight), _ptr(y), ws.ptr, ws.nbytes,
        _stream(stream)), "moe_combine")


def moe_shared_gate_weights(cfg, x, shared_gate, weights, stream=None) -> None:
    check(load_library().moe_shared_gate_weights(
        ctypes.byref(cfg), _ptr(x, "x"), _ptr(shared_gate, "shared_gate"),
        _ptr(weights, "weights"), _stream(stream)), "moe_shared_gate_weights")


def moe_balance_loss(cfg, counts, drops, mean_prob, alpha: float, loss, stream=None) -> None:
    check(load_library().moe_balance_loss(
        ctypes.byref(cfg), _ptr(counts, "counts"), _ptr(drops), _ptr(mean_prob, "mean_prob"),
        float(alpha), _ptr(loss, "loss"), _stream(stream)), "moe_balance_loss")


def moe_layer_forward(cfg, x, w_router, router_bias, score_bias, w_gate, w_up, w_down, ws_gate,
                      ws_up, ws_down, shared_gate, scales, y, topk_idx, topk_w, counts, drops,
                      mean_prob, ws: Workspace, stream=None) -> None:
    check(load_library().moe_layer_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(score_bias),
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down),
        _ptr(shared_gate), _scales_ref(scales), _ptr(y),
        _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(drops), _ptr(mean_prob), ws.ptr,
        ws.nbytes, _stream(stream)), "moe_layer_forward")


def _host_ptr(t: torch.Tensor, name: str, dtype: torch.dtype, numel: int):
    if t.is_cuda or not t.is_contiguous() or t.dtype != dtype or t.numel() != numel:
        raise ValueError(f"{name} must be a contiguous host tensor of {numel} {dtype}")
    return t.data_ptr()


def moe_layer_forward_host(cfg, x_host, x, w_router, router_bias, score_bias, w_gate, w_up,
                           w_down, ws_gate, ws_up, ws_down, shared_gate, scales, y, y_host,
                           topk_idx, topk_w, counts, drops, mean_prob, ws: Workspace,
                           stream=None) -> None:
    """moe_layer_forward with x read from and y written to host tensors (the
    copies run on ``stream``; pin both for them to be asynchronous)."""
    n = cfg.T * cfg.d_model
    check(load_library().moe_layer_forward_host(
        ctypes.byref(cfg), _host_ptr(x_host, "x_host", x.dtype, n), _ptr(x), _ptr(w_router),
        _ptr(router_bias), _ptr(score_bias), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
        _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), _ptr(shared_gate), _scales_ref(scales),
        _ptr(y), _host_ptr(y_host, "y_host", y.dtype, n), _ptr(topk_idx), _ptr(topk_w),
        _ptr(counts), _ptr(drops), _ptr(mean_prob), ws.ptr, ws.nbytes, _stream(stream)),
        "moe_layer_forward_host")


def moe_layer_forward_profiled(cfg, x, w_router, router_bias, score_bias, w_gate, w_up, w_down,
                               ws_gate, ws_up, ws_down, shared_gate, scales, y, topk_idx, topk_w,
                               counts, drops, mean_prob, ws: Workspace, stage_events,
                               stream=None) -> int:
    """moe_layer_forward recording ``stage_events`` (MOE_NUM_STAGES + 1
    torch.cuda.Event with timing, already recorded once so that they exist)
    before each stage; returns the number of kernels the call launched."""
    if len(stage_events) != B.MOE_NUM_STAGES + 1:
        raise ValueError("need MOE_NUM_STAGES + 1 events")
    arr = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
    n = ctypes.c_int32(0)
    check(load_library().moe_layer_forward_profiled(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(score_bias),
        _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), _ptr(shared_gate),
        _scales_ref(scales), _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(drops),
        _ptr(mean_prob), ws.ptr, ws.nbytes, _stream(stream), arr, ctypes.byref(n)),
        "moe_layer_forward_profiled")
    return n.value


def moe_get_error(ws: Workspace, stream=None) -> int:
    """Synchronises the stream; returns the workspace status code (0 = OK)."""
    return load_library().moe_get_error(ws.ptr, _stream(stream))


# ---------------------------------------------------------------------------
# Output-allocating conveniences
# ---------------------------------------------------------------------------

def _i32(n, device):
    return torch.empty(n, dtype=torch.int32, device=device)


def _f32(n, device):
    return torch.empty(n, dtype=torch.float32, device=device)


def route(cfg, x, w_router, router_bias=None, ws: Optional[Workspace] = None,
          want_logits=True, score_bias=None) -> Dict[str, torch.Tensor]:
    dev = x.device
    ws = ws or Workspace(cfg, dev)
    T, E, k = cfg.T, cfg.n_experts, cfg.top_k
    out = {"topk_idx": _i32((T, k), dev), "topk_w": _f32((T, k), dev),
           "mean_prob": _f32(E, dev)}
    out["logits"] = _f32((T, E), dev) if want_logits else None
    moe_router_topk(cfg, x, w_router, router_bias, score_bias, out["logits"], out["topk_idx"],
                    out["topk_w"], out["mean_prob"], ws)
    return out


def topk_from_logits(cfg, logits, ws: Optional[Workspace] = None,
                     score_bias=None) -> Dict[str, torch.Tensor]:
    dev = logits.device
    ws = ws or Workspace(cfg, dev)
    T, E, k = cfg.T, cfg.n_experts, cfg.top_k
    out = {"topk_idx": _i32((T, k), dev), "topk_w": _f32((T, k), dev),
           "mean_prob": _f32(E, dev)}
    moe_topk_from_logits(cfg, logits, score_bias, out["topk_idx"], out["topk_w"],
                         out["mean_prob"], ws)
    return out


def dispatch(cfg, topk_idx, ws: Optional[Workspace] = None) -> Dict[str, torch.Tensor]:
    dev = topk_idx.device
    ws = ws or Workspace(cfg, dev)
    E, A = cfg.n_experts, cfg.T * cfg.top_k
    out = {"counts": _i32(E, dev), "drops": _i32(E, dev), "offsets": _i32(E + 1, dev),
           "perm": _i32(max(A, 1), dev), "drop_mask": torch.empty(max(A, 1), dtype=torch.uint8,
                                                                   device=dev)}
    moe_dispatch(cfg, topk_idx, out["counts"], out["drops"], out["offsets"], out["perm"],
                 out["drop_mask"], ws)
    return out


@dataclass
class LayerWeights:
    w_router: torch.Tensor
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    router_bias: Optional[torch.Tensor] = None
    ws_gate: Optional[torch.Tensor] = None
    ws_up: Optional[torch.Tensor] = None
    ws_down: Optional[torch.Tensor] = None
    score_bias: Optional[torch.Tensor] = None
    shared_gate: Optional[torch.Tensor] = None
    scales: Optional[WeightScales] = None     # E4M3 expert weights only

    @classmethod
    def from_inputs(cls, inputs) -> "LayerWeights":
        return cls(inputs["w_router"], inputs["w_gate"], inputs["w_up"], inputs["w_down"],
                   inputs.get("router_bias"), inputs.get("ws_gate"), inputs.get("ws_up"),
                   inputs.get("ws_down"), inputs.get("score_bias"), inputs.get("shared_gate"),
                   WeightScales.from_inputs(inputs))


def layer_forward_host(cfg, x_host: torch.Tensor, w: LayerWeights, ws: Workspace,
                       x: torch.Tensor, y: torch.Tensor, y_host: torch.Tensor,
                       stream=None) -> torch.Tensor:
    """One layer call on host token rows: x_host is copied into the device
    staging buffer x, the layer writes y, and y is copied into y_host, all
    enqueued on ``stream``; y_host is valid once the stream has reached the
    end of the call.  Statistics are not returned."""
    moe_layer_forward_host(cfg, x_host, x, w.w_router, w.router_bias, w.score_bias, w.w_gate,
                           w.w_up, w.w_down, w.ws_gate, w.ws_up, w.ws_down, w.shared_gate,
                           w.scales, y, y_host, None, None, None, None, None, ws, stream)
    return y_host


def layer_forward(cfg, x, w: LayerWeights, ws: Optional[Workspace] = None,
                  y: Optional[torch.Tensor] = None, stats: bool = True,
                  stream=None) -> Dict[str, torch.Tensor]:
    dev = x.device
    ws = ws or Workspace(cfg, dev)
    T, E, k, d = cfg.T, cfg.n_experts, cfg.top_k, cfg.d_model
    out = {"y": y if y is not None else torch.empty((T, d), dtype=out_dtype(cfg), device=dev)}
    if stats:
        out.update(counts=_i32(E, dev), drops=_i32(E, dev), mean_prob=_f32(E, dev))
        if cfg.routing == B.MOE_ROUTE_TOKEN_CHOICE:   # expert choice has no per-token top-k
            out.update(topk_idx=_i32((T, k), dev), topk_w=_f32((T, k), dev))
    g = out.get
    moe_layer_forward(cfg, x, w.w_router, w.router_bias, w.score_bias, w.w_gate, w.w_up,
                      w.w_down, w.ws_gate, w.ws_up, w.ws_down, w.shared_gate, w.scales, out["y"],
                      g("topk_idx"),
                      g("topk_w"), g("counts"), g("drops"), g("mean_prob"), ws, stream)
    return out
