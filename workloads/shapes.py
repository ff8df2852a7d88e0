"""The five MoE layer shapes the library is tested and measured on.

Each shape follows a model configuration that the pages describe:

* ``tiny`` - a 4-expert top-2 layer small enough for pure-Python checks.
* ``mixtral`` - Mixtral-8x7B: d_model 4096, 8 experts of SwiGLU d_ff 14336,
  top-2, softmax gating with renormalisation ("10. 混合专家 MoE：总参数与激活参数",
  niuwancheng.cn, sections "把一个大 FFN 换成一组小 FFN" and
  "总参数和激活参数怎样算").
* ``dsv3_prefill`` / ``dsv3_decode`` - DeepSeek-V3: d_model 7168, 256 routed
  experts of d_ff 2048, top-8, one always-on shared expert, sigmoid gating,
  renormalisation times routed_scaling_factor 2.5 (same page, sections
  "路由器怎样选专家：top-k 与两种门控" and "细粒度专家与共享专家").
* ``dsv3_prefill_noaux`` - the same layer routed the way DeepSeek-V3 routes:
  ranking by sigmoid score plus a selection-only bias, with 8 expert groups of
  which each token may use 4 (same page, "DeepSeek-V3 的无辅助损失偏置").
* ``dsv3_decode_fp8`` / ``dsv3_prefill_fp8`` - the DeepSeek-V3 layers with the
  expert weights stored as FP8 E4M3 codes and one scale per output channel
  (same page, "推理时": DeepSeek-V3 ships FP8 weights).
* ``switch_expert_choice`` - the Switch-shaped layer routed by expert choice:
  each of the 64 experts takes the 256 tokens it scores highest (the
  amazingdata.cn article on MoE routing, paragraph on expert choice).
* ``switch`` - a Switch-Transformer-style top-1 layer with an expert capacity
  of ceil(T/E x 1.25) and token dropping (same page, section
  "负载不均：路由坍缩与丢 token"), with a Zipf-skewed router bias so that the
  hottest experts overflow.

The shapes only fix sizes, gating options and dtypes.
"""

from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int            # tokens in the batch
    d: int            # d_model
    E: int            # routed experts
    k: int            # experts per token (num_experts_per_tok)
    F: int            # routed expert SwiGLU d_ff (moe_intermediate_size)
    F_s: int          # shared expert d_ff, 0 = no shared expert
    gate: str         # "softmax" or "sigmoid"
    renormalize: bool
    rsf: float        # routed_scaling_factor
    capacity_factor: Optional[float]   # None = unlimited capacity
    zipf_s: Optional[float]            # router bias skew exponent, None = no bias
    dtype: str        # "fp32" or "bf16" (activations and weights)
    n_group: int = 0  # expert groups for group-limited selection (0 = none)
    topk_group: int = 0               # groups kept per token
    score_bias_std: Optional[float] = None   # selection-only score bias ~ N(0, std^2)
    shared_gate: bool = False         # per-token sigmoid gate on the shared expert
    weight_format: str = "act"        # "act" (weights in dtype) or "fp8" (E4M3 + row scales)
    routing: str = "token"            # "token" (top-k per token) or "expert" (top-C per expert)

    def with_tokens(self, T: int) -> "MoEShape":
        return replace(self, T=T)

    @property
    def assignments(self) -> int:
        return self.T * self.k


SHAPES = {
    "tiny": MoEShape("tiny", T=64, d=128, E=4, k=2, F=256, F_s=0, gate="softmax",
                     renormalize=True, rsf=1.0, capacity_factor=None, zipf_s=None,
                     dtype="fp32"),
    "mixtral": MoEShape("mixtral", T=4096, d=4096, E=8, k=2, F=14336, F_s=0,
                        gate="softmax", renormalize=True, rsf=1.0,
                        capacity_factor=None, zipf_s=None, dtype="bf16"),
    "dsv3_prefill": MoEShape("dsv3_prefill", T=8192, d=7168, E=256, k=8, F=2048,
                             F_s=2048, gate="sigmoid", renormalize=True, rsf=2.5,
                             capacity_factor=None, zipf_s=None, dtype="bf16"),
    "switch": MoEShape("switch", T=16384, d=2048, E=64, k=1, F=8192, F_s=0,
                       gate="softmax", renormalize=False, rsf=1.0,
                       capacity_factor=1.25, zipf_s=1.2, dtype="bf16"),
    # DeepSeek-V3's own router ("DeepSeek-V3 的无辅助损失偏置"): rank by
    # s + b with a selection-only bias, 8 groups of 32 experts, 4 kept
    "dsv3_prefill_noaux": MoEShape("dsv3_prefill_noaux", T=8192, d=7168, E=256, k=8, F=2048,
                                   F_s=2048, gate="sigmoid", renormalize=True, rsf=2.5,
                                   capacity_factor=None, zipf_s=None, dtype="bf16",
                                   n_group=8, topk_group=4, score_bias_std=0.02),
    "dsv3_decode": MoEShape("dsv3_decode", T=64, d=7168, E=256, k=8, F=2048,
                            F_s=2048, gate="sigmoid", renormalize=True, rsf=2.5,
                            capacity_factor=None, zipf_s=None, dtype="bf16"),
    # the Switch-shaped layer routed by expert choice: each expert takes
    # C = T * k / E = 256 tokens (the amazingdata.cn routing article, paragraph
    # on expert choice: each expert takes a fixed number of its best tokens)
    "switch_expert_choice": MoEShape("switch_expert_choice", T=16384, d=2048, E=64, k=1,
                                     F=8192, F_s=0, gate="softmax", renormalize=False, rsf=1.0,
                                     capacity_factor=None, zipf_s=None, dtype="bf16",
                                     routing="expert"),
    # the same layers with E4M3 expert weights (one scale per output channel)
    "dsv3_decode_fp8": MoEShape("dsv3_decode_fp8", T=64, d=7168, E=256, k=8, F=2048,
                                F_s=2048, gate="sigmoid", renormalize=True, rsf=2.5,
                                capacity_factor=None, zipf_s=None, dtype="bf16",
                                weight_format="fp8"),
    "dsv3_prefill_fp8": MoEShape("dsv3_prefill_fp8", T=8192, d=7168, E=256, k=8, F=2048,
                                 F_s=2048, gate="sigmoid", renormalize=True, rsf=2.5,
                                 capacity_factor=None, zipf_s=None, dtype="bf16",
                                 weight_format="fp8"),
}


def shape_by_name(name: str) -> MoEShape:
    return SHAPES[name]
