"""Routed ReLU^2 mixture-of-experts layer (NemotronH-style) for GB300 (sm_103a).

The compute lives in the CUDA library ``lib/libmoe_gb300.so`` behind the C ABI
of ``include/moe_gb300.h``; this package is its thin binding.
"""
from ._native import (EXPORTS, LIB_PATH, MOE_DEVERR_EXPERT_ID, MOE_DEVERR_NONFINITE,
                      MOE_DEVERR_SCHEDULE, MOE_DT_BF16, MOE_DT_F32, MOE_DT_NVFP4, MoEError,
                      MoeConfig, MoeWeights, load)
from .layer import (GRAD_FIELDS, MoEBlock, MoELayer, Weights, backward_workspace_bytes, backward_workspace_region,
                    moe_block_backward,
                    moe_layer_backward, new_backward_workspace, config_from, make_config, moe_clear_device_error,
                    moe_dispatch, moe_experts_down, moe_experts_down_combine, moe_experts_up, moe_get_device_error,
                    moe_block_forward, moe_latent_down, moe_layer_forward, moe_layer_forward_host, moe_router,
                    moe_router_noalloc, moe_shared, new_workspace, nvfp4_act_terms_for, set_nvfp4_act_terms,
                    sparse_down_bytes, sparse_down_layout, workspace_bytes,
                    workspace_region)

__all__ = [
    "EXPORTS", "LIB_PATH", "MOE_DEVERR_EXPERT_ID", "MOE_DEVERR_NONFINITE", "MOE_DEVERR_SCHEDULE",
    "MOE_DT_BF16", "MOE_DT_F32", "MOE_DT_NVFP4", "MoEError", "MoeConfig", "MoeWeights", "load",
    "GRAD_FIELDS", "MoEBlock", "MoELayer", "Weights", "backward_workspace_bytes", "backward_workspace_region",
    "moe_block_backward",
    "moe_layer_backward", "new_backward_workspace", "config_from", "make_config", "moe_clear_device_error", "moe_dispatch",
    "moe_block_forward", "moe_experts_down", "moe_experts_down_combine", "moe_experts_up", "moe_get_device_error",
    "moe_latent_down",
    "moe_layer_forward", "moe_layer_forward_host", "moe_router", "moe_router_noalloc", "moe_shared", "new_workspace",
    "nvfp4_act_terms_for", "set_nvfp4_act_terms", "sparse_down_bytes", "sparse_down_layout", "workspace_bytes",
    "workspace_region",
]
