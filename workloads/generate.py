"""Seeded synthetic tensors for an MoE layer shape.

Recipe (one torch.Generator stream per tensor, seeded from the tensor's name):

* x        ~ N(0, 1)          [T, d]
* w_router ~ N(0, 1/d)        [E, d]      (nn.Linear orientation: out x in)
* w_gate   ~ N(0, 1/d)        [E, F, d]   one stream per expert
* w_up     ~ N(0, 1/d)        [E, F, d]
* w_down   ~ N(0, 1/F)        [E, d, F]
* ws_gate, ws_up ~ N(0, 1/d)  [F_s, d]    shared expert (when F_s > 0)
* ws_down  ~ N(0, 1/F_s)      [d, F_s]
* router_bias (Zipf-skewed shapes only): b_e = -s * ln(e + 1), the log of an
  unnormalised Zipf(s) mass, so expert 0 is the hottest.  The normaliser of
  the Zipf pmf would cancel under softmax and under the argmax, so it is left
  out.
* score_bias (shapes with score_bias_std): ~ N(0, std^2) [E] fp32, standing in
  for a selection-only bias after some training steps of +-gamma.
* shared_gate (shapes with a gated shared expert) ~ N(0, 1/d) [d].
* FP8 shapes: each expert weight above is drawn the same way in float32 and
  stored as E4M3 codes (torch.float8_e4m3fn, round to nearest even) of
  w / s with s = max|w_row| / 448 per output row, plus the fp32 row scales
  (w_gate_scale, w_up_scale, w_down_scale, ws_*_scale).

Values are drawn in float32 and then cast to the shape's dtype (bf16 or fp32).
This module holds no routing or expert arithmetic.
"""

from __future__ import annotations

import math
import zlib
from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np
import torch

from .shapes import MoEShape

_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


def tensor_seed(seed_base: int, name: str) -> int:
    """Deterministic per-tensor seed: CRC32 of "<seed_base>:<name>"."""
    return zlib.crc32(f"{seed_base}:{name}".encode()) & 0x7FFFFFFF


def _normal(shape, std: float, name: str, seed_base: int, device, dtype) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(tensor_seed(seed_base, name))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


E4M3_MAX = 448.0


def quantize_rows_e4m3(w: torch.Tensor):
    """(codes, scales): E4M3 codes of w / s and the per-row scales
    s = max|w_row| / 448 (1 for an all-zero row)."""
    w = w.float()
    s = w.abs().amax(dim=-1) / E4M3_MAX
    s = torch.where(s > 0, s, torch.ones_like(s))
    q = (w / s.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q, s


def _weight(shape_, std, name, seed, device, dt, fp8: bool):
    w = _normal(shape_, std, name, seed, device, torch.float32)
    if fp8:
        return quantize_rows_e4m3(w)
    return w.to(dt), None


def make_inputs(shape: MoEShape, device="cpu", seed: int = 0,
                with_experts: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """All tensors of one layer instance, on ``device``.

    Returns a dict with keys x, w_router, router_bias, w_gate, w_up, w_down,
    ws_gate, ws_up, ws_down (absent parts are None).
    """
    dt = _DTYPES[shape.dtype]
    T, d, E, F, Fs = shape.T, shape.d, shape.E, shape.F, shape.F_s
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _normal((T, d), 1.0, "x", seed, device, dt)
    out["w_router"] = _normal((E, d), 1.0 / math.sqrt(d), "w_router", seed, device, dt)
    if shape.zipf_s is not None:
        e = torch.arange(E, dtype=torch.float64)
        out["router_bias"] = (-shape.zipf_s * torch.log(e + 1.0)).to(torch.float32).to(device)
    else:
        out["router_bias"] = None
    if getattr(shape, "score_bias_std", None):
        out["score_bias"] = _normal((E,), shape.score_bias_std, "score_bias", seed, device,
                                    torch.float32)
    else:
        out["score_bias"] = None
    if with_experts:
        fp8 = getattr(shape, "weight_format", "act") == "fp8"
        wdt = torch.float8_e4m3fn if fp8 else dt
        wg = torch.empty((E, F, d), dtype=wdt, device=device)
        wu = torch.empty((E, F, d), dtype=wdt, device=device)
        wd = torch.empty((E, d, F), dtype=wdt, device=device)
        if fp8:
            sg = torch.empty((E, F), dtype=torch.float32, device=device)
            su = torch.empty((E, F), dtype=torch.float32, device=device)
            sd = torch.empty((E, d), dtype=torch.float32, device=device)
        for e in range(E):
            q, s = _weight((F, d), 1.0 / math.sqrt(d), f"w_gate.{e}", seed, device, dt, fp8)
            wg[e] = q
            if fp8:
                sg[e] = s
            q, s = _weight((F, d), 1.0 / math.sqrt(d), f"w_up.{e}", seed, device, dt, fp8)
            wu[e] = q
            if fp8:
                su[e] = s
            q, s = _weight((d, F), 1.0 / math.sqrt(F), f"w_down.{e}", seed, device, dt, fp8)
            wd[e] = q
            if fp8:
                sd[e] = s
        out["w_gate"], out["w_up"], out["w_down"] = wg, wu, wd
        if fp8:
            out["w_gate_scale"], out["w_up_scale"], out["w_down_scale"] = sg, su, sd
        if Fs > 0:
            for key, shp, std in (("ws_gate", (Fs, d), 1.0 / math.sqrt(d)),
                                  ("ws_up", (Fs, d), 1.0 / math.sqrt(d)),
                                  ("ws_down", (d, Fs), 1.0 / math.sqrt(Fs))):
                q, s = _weight(shp, std, key, seed, device, dt, fp8)
                out[key] = q
                if fp8:
                    out[key + "_scale"] = s
        else:
            out["ws_gate"] = out["ws_up"] = out["ws_down"] = None
        out["shared_gate"] = None
        if Fs > 0 and getattr(shape, "shared_gate", False):
            out["shared_gate"] = _normal((d,), 1.0 / math.sqrt(d), "shared_gate", seed, device, dt)
    return out


def to_f64(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact widening of a bf16/fp32 tensor (any device) to a float64 array."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


@dataclass
class ExpertWeights:
    """Lazy per-expert float64 view of the expert weight tensors.

    ``weights[e]`` returns (w_gate_e [F,d], w_up_e [F,d], w_down_e [d,F]) as
    float64 arrays, converting one expert at a time so that a 22 GB bf16 layer
    never has to exist as a 90 GB float64 copy.
    """
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor

    def __len__(self) -> int:
        return self.w_gate.shape[0]

    def __getitem__(self, e: int):
        return to_f64(self.w_gate[e]), to_f64(self.w_up[e]), to_f64(self.w_down[e])


def shared_weights(inputs) -> Optional[tuple]:
    if inputs.get("ws_gate") is None:
        return None
    return to_f64(inputs["ws_gate"]), to_f64(inputs["ws_up"]), to_f64(inputs["ws_down"])
