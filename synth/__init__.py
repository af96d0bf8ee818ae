"""Seeded synthetic workloads for the routed ReLU^2 MoE layer (shapes + random inputs)."""
from .configs import (BF16, F32, NVFP4, MoEShape, NANO_DECODE, NANO_DECODE_SPARSE, NANO_PREFILL,
                      ROUTER_ONLY_GROUPED, SUPER_LATENT, SUPER_NVFP4, SUPER_NVFP4_SPARSE, TINY_FP32,
                      WORKLOADS, scaled)
from .generate import (make_calibration_x, make_norm_weight, make_weights, make_x, quantize_nvfp4,
                       router_params, zipf_offsets, zipf_targets)

__all__ = [
    "BF16", "F32", "NVFP4", "MoEShape", "NANO_DECODE", "NANO_DECODE_SPARSE", "NANO_PREFILL", "ROUTER_ONLY_GROUPED",
    "SUPER_LATENT", "SUPER_NVFP4", "SUPER_NVFP4_SPARSE", "TINY_FP32", "WORKLOADS", "scaled", "make_calibration_x", "make_norm_weight",
    "make_weights", "make_x", "quantize_nvfp4", "router_params", "zipf_offsets", "zipf_targets",
]
