"""Single-GPU MoE FFN layer forward for NVIDIA B300 (sm_103a).

The compute path is libmoe_b300.so (hand-written CUDA kernels behind the C ABI
in include/moe_b300.h); this package only marshals torch tensors into it.
"""

from ._binding import MoEConfig, MoEError, load_library  # noqa: F401
from .api import (  # noqa: F401
    LayerWeights, Workspace, config_from_shape, dispatch, layer_forward, make_config,
    moe_capacity, moe_combine, moe_dispatch, moe_get_error, moe_grouped_swiglu,
    moe_layer_forward, moe_layer_forward_profiled, moe_router_topk, moe_topk_from_logits,
    moe_update_score_bias, moe_version, moe_workspace_size, route, topk_from_logits,
    moe_shared_gate_weights, moe_balance_loss, moe_expert_choice_capacity,
    moe_expert_choice_from_logits, expert_choice_from_logits, layer_forward_host,
    moe_layer_forward_host,
)
