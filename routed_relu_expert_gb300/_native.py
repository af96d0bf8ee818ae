"""ctypes binding of the C ABI declared in include/moe_gb300.h.

Argument marshalling only: every step of the layer runs in the CUDA library.
If the shared library is missing the import of any entry point fails loudly;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(6)
MOE_DEVERR_EXPERT_ID, MOE_DEVERR_NONFINITE, MOE_DEVERR_SCHEDULE, MOE_DEVERR_TIMEOUT, MOE_DEVERR_RANGE = 1, 2, 4, 8, 16
MOE_DT_F32, MOE_DT_BF16, MOE_DT_NVFP4 = 0, 1, 2
MOE_NOALLOC_MAX_ROUTER_ELEMS = 131072
MOE_NOALLOC_MAX_SPLIT_ELEMS = 7340032
(MOE_WS_COUNTS, MOE_WS_OFFSETS, MOE_WS_ROUTE_TOKEN, MOE_WS_ROUTE_SLOT, MOE_WS_TOKEN_SLOT_ROW, MOE_WS_TOPK_IDS,
 MOE_WS_TOPK_W, MOE_WS_LOGITS, MOE_WS_SCORES, MOE_WS_X_LATENT, MOE_WS_X_PACKED, MOE_WS_H, MOE_WS_X_TERMS,
 MOE_WS_X_TERM_SCALES, MOE_WS_X_ROW_SCALES, MOE_WS_H_TERMS, MOE_WS_H_TERM_SCALES, MOE_WS_H_ROW_SCALES,
 MOE_WS_X_NORM) = range(19)
ACT_TERMS_MAX = 4
MOE_BWS_DU, MOE_BWS_DA, MOE_BWS_DZ, MOE_BWS_DX_LATENT, MOE_BWS_DA_SHARED, MOE_BWS_DY_LATENT = range(6)


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("d_model", ctypes.c_int32),
        ("d_latent", ctypes.c_int32),
        ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("n_group", ctypes.c_int32),
        ("topk_group", ctypes.c_int32),
        ("d_expert", ctypes.c_int32),
        ("d_shared", ctypes.c_int32),
        ("norm_topk_prob", ctypes.c_int32),
        ("routed_scaling_factor", ctypes.c_float),
        ("act_dtype", ctypes.c_int32),
        ("expert_dtype", ctypes.c_int32),
    ]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_router", "router_bias", "w_lat_down", "w_lat_up", "w_up", "w_down",
        "w_up_sf", "w_down_sf", "w_up_gs", "w_down_gs", "w_sh_up", "w_sh_down", "w_down_g", "w_down_g_sf")]


class MoeGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "d_router", "d_lat_down", "d_lat_up", "d_up", "d_down", "d_sh_up", "d_sh_down", "d_norm_w")]


EXPORTS = (
    "moe_version", "moe_status_string", "moe_check_config", "moe_workspace_bytes", "moe_router",
    "moe_dispatch", "moe_experts_up", "moe_experts_down", "moe_experts_down_combine", "moe_latent_down", "moe_shared",
    "moe_layer_forward", "moe_get_device_error", "moe_clear_device_error", "moe_layer_forward_host",
    "moe_launch_count", "moe_router_noalloc", "moe_workspace_region", "moe_set_nvfp4_act_terms",
    "moe_nvfp4_act_terms_for", "moe_block_forward", "moe_sparse_down_bytes", "moe_sparse_down_layout",
    "moe_backward_workspace_bytes", "moe_layer_backward", "moe_block_backward", "moe_backward_workspace_region",
)

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run python -m routed_relu_expert_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I32 = ctypes.c_int32
    S = ctypes.c_size_t
    CFG = ctypes.POINTER(MoeConfig)
    W = ctypes.POINTER(MoeWeights)
    sig = {
        "moe_version": (I32, []),
        "moe_status_string": (ctypes.c_char_p, [I32]),
        "moe_check_config": (I32, [CFG]),
        "moe_workspace_bytes": (S, [CFG, I32]),
        "moe_router": (I32, [CFG, I32, P, P, P, P, P, P, P, P, S, P]),
        "moe_dispatch": (I32, [CFG, I32, P, P, P, P, P, P, P, P, P, S, P]),
        "moe_experts_up": (I32, [CFG, I32, P, P, P, P, W, P, P, S, P]),
        "moe_experts_down": (I32, [CFG, I32, P, P, P, P, P, W, P, P, S, P]),
        "moe_experts_down_combine": (I32, [CFG, I32, P, P, P, P, P, P, W, P, P, S, P]),
        "moe_latent_down": (I32, [CFG, I32, P, W, P, P, S, P]),
        "moe_shared": (I32, [CFG, I32, P, W, P, P, P, S, P]),
        "moe_layer_forward": (I32, [CFG, I32, P, W, P, P, P, P, P, P, S, P]),
        "moe_block_forward": (I32, [CFG, I32, P, P, ctypes.c_float, W, P, P, P, P, P, P, P, S, P]),
        "moe_sparse_down_bytes": (I32, [CFG, ctypes.POINTER(S), ctypes.POINTER(S)]),
        "moe_sparse_down_layout": (I32, [CFG, W, P, P, P]),
        "moe_backward_workspace_bytes": (S, [CFG, I32]),
        "moe_backward_workspace_region": (I32, [CFG, I32, I32, ctypes.POINTER(S), ctypes.POINTER(S)]),
        "moe_layer_backward": (I32, [CFG, I32, P, W, P, P, P, P, P, ctypes.POINTER(MoeGrads), P, S, P, S, P]),
        "moe_block_backward": (I32, [CFG, I32, P, P, ctypes.c_float, P, W, P, P, P, P, P,
                                     ctypes.POINTER(MoeGrads), P, S, P, S, P]),
        "moe_get_device_error": (I32, [P, P, ctypes.POINTER(I32)]),
        "moe_clear_device_error": (I32, [P, P]),
        "moe_layer_forward_host": (I32, [CFG, I32, P, P, W, P, P, P, S, P]),
        "moe_launch_count": (ctypes.c_int64, []),
        "moe_router_noalloc": (I32, [CFG, I32, P, P, P, P, P, P]),
        "moe_workspace_region": (I32, [CFG, I32, I32, ctypes.POINTER(S), ctypes.POINTER(S)]),
        "moe_set_nvfp4_act_terms": (I32, [I32]),
        "moe_nvfp4_act_terms_for": (I32, [I32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().moe_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, where)
