"""B300-native (sm_103a) forward pass of one Mixture-of-Experts layer.

The compute path is libmoe.so (C ABI in include/moe.h); `binding` marshals
torch tensors into it.  `inputs` draws the seeded synthetic workloads.
"""
from .binding import (  # noqa: F401
    MoEError, MoELayer, Workspace, lib, make_shape, moe_check_device_status, moe_clear_device_status,
    moe_combine, moe_combine_bf16, moe_expert_down, moe_expert_up, moe_forward, moe_forward_a_path, moe_forward_bf16,
    moe_permute, moe_prepare_weights, moe_route, moe_router_logits, moe_row_capacity, moe_selftest_timeout, moe_token_round,
    moe_topk_gating, moe_workspace_bytes, moe_workspace_layout, status_string,
)
