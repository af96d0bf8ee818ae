"""Python entry points with the C ABI's names, over torch-allocated device memory.

Each function checks tensor placement, takes data pointers and the current
CUDA stream, and calls the library; nothing here computes any part of the
layer.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import torch

from . import _native as N

_DT = {"f32": N.MOE_DT_F32, "bf16": N.MOE_DT_BF16, "nvfp4": N.MOE_DT_NVFP4}


def make_config(d_model: int, n_experts: int, top_k: int, d_expert: int, *, d_latent: int = 0,
                n_group: int = 1, topk_group: int = 1, d_shared: int = 0, norm_topk_prob: int = 1,
                routed_scaling_factor: float = 1.0, act_dtype: int = N.MOE_DT_BF16,
                expert_dtype: int = N.MOE_DT_BF16) -> N.MoeConfig:
    return N.MoeConfig(d_model, d_latent, n_experts, top_k, n_group, topk_group, d_expert, d_shared,
                       norm_topk_prob, float(routed_scaling_factor), act_dtype, expert_dtype)


def config_from(shape) -> N.MoeConfig:
    """Config from any object carrying the layer's shape attributes."""
    return make_config(shape.d_model, shape.n_experts, shape.top_k, shape.d_expert,
                       d_latent=shape.d_latent, n_group=shape.n_group, topk_group=shape.topk_group,
                       d_shared=shape.d_shared, norm_topk_prob=shape.norm_topk_prob,
                       routed_scaling_factor=shape.routed_scaling_factor, act_dtype=shape.act_dtype,
                       expert_dtype=shape.expert_dtype)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _hp(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("host tensor must be a contiguous CPU tensor")
    return ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Weights:
    """Keeps a layer's device tensors alive and exposes them as moe_weights_t."""

    FIELDS = ("w_router", "router_bias", "w_lat_down", "w_lat_up", "w_up", "w_down", "w_up_sf",
              "w_down_sf", "w_up_gs", "w_down_gs", "w_sh_up", "w_sh_down", "w_down_g", "w_down_g_sf")
    ALIASES = {"router_bias": "bias", "w_up": "w_up_q", "w_down": "w_down_q"}

    def __init__(self, tensors: Dict[str, torch.Tensor]):
        self.tensors = {}
        vals = {}
        for f in self.FIELDS:
            t = tensors.get(f)
            if t is None and f in self.ALIASES:
                t = tensors.get(self.ALIASES[f])
            if t is not None:
                self.tensors[f] = t
                vals[f] = _p(t)
        self.struct = N.MoeWeights(**{f: vals.get(f) for f in self.FIELDS})

    @property
    def ref(self):
        return ctypes.byref(self.struct)


def workspace_bytes(cfg: N.MoeConfig, T: int) -> int:
    return int(N.load().moe_workspace_bytes(ctypes.byref(cfg), int(T)))


def new_workspace(cfg: N.MoeConfig, T: int, device="cuda") -> torch.Tensor:
    n = workspace_bytes(cfg, T)
    if n == 0 and T > 0:
        N.check(N.load().moe_check_config(ctypes.byref(cfg)), "moe_workspace_bytes")
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    ws[:256].zero_()    # the header: error word clear, no schedule yet
    return ws


def set_nvfp4_act_terms(n: int) -> int:
    """How NVFP4 experts take their activations (-1: the measured default;
    0: FP16 path; 1..4: NVFP4 terms on the FP4 tensor path); returns the
    previous setting."""
    prev = int(N.load().moe_set_nvfp4_act_terms(int(n)))
    if prev < -1:
        raise ValueError(f"activation terms must be -1..4, got {n}")
    return prev


def nvfp4_act_terms_for(T: int) -> int:
    """Activation terms an NVFP4 layer of T tokens uses now (0: FP16 path)."""
    return int(N.load().moe_nvfp4_act_terms_for(int(T)))


def workspace_region(cfg: N.MoeConfig, T: int, region: int):
    """(byte offset, bytes) of one of the route tables in a workspace for T tokens."""
    off, n = ctypes.c_size_t(0), ctypes.c_size_t(0)
    N.check(N.load().moe_workspace_region(ctypes.byref(cfg), int(T), int(region), ctypes.byref(off),
                                          ctypes.byref(n)), "moe_workspace_region")
    return int(off.value), int(n.value)


def _ws(ws: torch.Tensor):
    return _p(ws), ctypes.c_size_t(ws.numel())


# ---------------------------------------------------------------------------
def moe_router(cfg, x, w_router, bias, ids, topw, ws, logits=None, scores=None, stream=None):
    T = x.shape[0]
    w, n = _ws(ws)
    N.check(N.load().moe_router(ctypes.byref(cfg), T, _p(x), _p(w_router), _p(bias), _p(logits), _p(scores),
                                _p(ids), _p(topw), w, n, _s(stream)), "moe_router")


def moe_router_noalloc(cfg, x, w_router, bias, ids, topw, stream=None):
    """Router with no workspace (scratch in the library's static device array)."""
    N.check(N.load().moe_router_noalloc(ctypes.byref(cfg), x.shape[0], _p(x), _p(w_router), _p(bias), _p(ids),
                                        _p(topw), _s(stream)), "moe_router_noalloc")


def moe_dispatch(cfg, ids, counts, offsets, route_token, route_slot, token_slot_row, ws, x_e=None,
                 x_packed=None, stream=None):
    T = ids.shape[0]
    w, n = _ws(ws)
    N.check(N.load().moe_dispatch(ctypes.byref(cfg), T, _p(ids), _p(x_e), _p(counts), _p(offsets),
                                  _p(route_token), _p(route_slot), _p(token_slot_row), _p(x_packed), w, n,
                                  _s(stream)), "moe_dispatch")


def moe_experts_up(cfg, T, route_token, offsets, weights: Weights, h, ws, x_e=None, x_packed=None, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_experts_up(ctypes.byref(cfg), T, _p(x_e), _p(x_packed), _p(route_token), _p(offsets),
                                    weights.ref, _p(h), w, n, _s(stream)), "moe_experts_up")


def moe_experts_down_combine(cfg, T, h, offsets, route_token, route_slot, token_slot_row, topw,
                             weights: Weights, y_routed, ws, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_experts_down_combine(ctypes.byref(cfg), T, _p(h), _p(offsets), _p(route_token),
                                              _p(route_slot), _p(token_slot_row), _p(topw), weights.ref,
                                              _p(y_routed), w, n, _s(stream)), "moe_experts_down_combine")


def moe_experts_down(cfg, T, h, offsets, route_token, route_slot, topw, weights: Weights, u, ws, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_experts_down(ctypes.byref(cfg), T, _p(h), _p(offsets), _p(route_token), _p(route_slot),
                                      _p(topw), weights.ref, _p(u), w, n, _s(stream)), "moe_experts_down")


def moe_latent_down(cfg, x, weights: Weights, x_l, ws, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_latent_down(ctypes.byref(cfg), x.shape[0], _p(x), weights.ref, _p(x_l), w, n,
                                     _s(stream)), "moe_latent_down")


def moe_shared(cfg, x, weights: Weights, y, ws, y_routed=None, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_shared(ctypes.byref(cfg), x.shape[0], _p(x), weights.ref, _p(y_routed), _p(y), w, n,
                                _s(stream)), "moe_shared")


def moe_layer_forward(cfg, x, weights: Weights, y, ws, ids_out=None, topw_out=None, logits_out=None,
                      scores_out=None, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_layer_forward(ctypes.byref(cfg), x.shape[0], _p(x), weights.ref, _p(y), _p(ids_out),
                                       _p(topw_out), _p(logits_out), _p(scores_out), w, n, _s(stream)),
            "moe_layer_forward")


def sparse_down_bytes(cfg):
    """(values, scales) bytes of the group-major down weights of a configuration."""
    v, sc = ctypes.c_size_t(0), ctypes.c_size_t(0)
    N.check(N.load().moe_sparse_down_bytes(ctypes.byref(cfg), ctypes.byref(v), ctypes.byref(sc)),
            "moe_sparse_down_bytes")
    return int(v.value), int(sc.value)


def sparse_down_layout(cfg, weights: Weights, stream=None) -> Dict[str, torch.Tensor]:
    """The expert down weights re-laid group-major (w_down_g, and w_down_g_sf for
    NVFP4) by the library, as new device tensors."""
    nv, ns = sparse_down_bytes(cfg)
    dev = weights.tensors["w_down"].device
    out = {"w_down_g": torch.empty(nv, dtype=torch.uint8, device=dev)}
    if ns:
        out["w_down_g_sf"] = torch.empty(ns, dtype=torch.uint8, device=dev)
    N.check(N.load().moe_sparse_down_layout(ctypes.byref(cfg), weights.ref, _p(out["w_down_g"]),
                                            _p(out.get("w_down_g_sf")), _s(stream)), "moe_sparse_down_layout")
    return out


def moe_block_forward(cfg, x, norm_w, norm_eps: float, weights: Weights, out, ws, x_norm_out=None, ids_out=None,
                      topw_out=None, logits_out=None, scores_out=None, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_block_forward(ctypes.byref(cfg), x.shape[0], _p(x), _p(norm_w), ctypes.c_float(norm_eps),
                                       weights.ref, _p(out), _p(x_norm_out), _p(ids_out), _p(topw_out),
                                       _p(logits_out), _p(scores_out), w, n, _s(stream)),
            "moe_block_forward")


GRAD_FIELDS = ("d_router", "d_lat_down", "d_lat_up", "d_up", "d_down", "d_sh_up", "d_sh_down", "d_norm_w")


def _grads(grads: Optional[Dict[str, torch.Tensor]]) -> N.MoeGrads:
    grads = grads or {}
    for k in grads:
        if k not in GRAD_FIELDS:
            raise KeyError(f"unknown gradient {k}")
    return N.MoeGrads(**{f: _p(grads.get(f)) for f in GRAD_FIELDS})


def backward_workspace_bytes(cfg, T: int) -> int:
    return int(N.load().moe_backward_workspace_bytes(ctypes.byref(cfg), T))


def backward_workspace_region(cfg, T: int, region: int):
    """(byte offset, bytes) of a region of the backward scratch (MOE_BWS_*)."""
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    N.check(N.load().moe_backward_workspace_region(ctypes.byref(cfg), T, region, ctypes.byref(off),
                                                   ctypes.byref(nb)), "moe_backward_workspace_region")
    return int(off.value), int(nb.value)


def new_backward_workspace(cfg, T: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(backward_workspace_bytes(cfg, T), 256), dtype=torch.uint8, device=device)


def moe_layer_backward(cfg, x, weights: Weights, dy, ids, topw, scores, dx, grads, ws, bws, stream=None):
    """dx (FP32) and weight gradients (added to the FP32 tensors in ``grads``,
    keys from GRAD_FIELDS) of the forward whose state ``ws`` holds."""
    w, n = _ws(ws)
    b, nb = _ws(bws)
    g = _grads(grads)
    N.check(N.load().moe_layer_backward(ctypes.byref(cfg), x.shape[0], _p(x), weights.ref, _p(dy), _p(ids),
                                        _p(topw), _p(scores), _p(dx), ctypes.byref(g), w, n, b, nb, _s(stream)),
            "moe_layer_backward")


def moe_block_backward(cfg, x, norm_w, norm_eps: float, weights: Weights, dout, ids, topw, scores, dx, grads, ws,
                       bws, x_norm=None, stream=None):
    w, n = _ws(ws)
    b, nb = _ws(bws)
    g = _grads(grads)
    N.check(N.load().moe_block_backward(ctypes.byref(cfg), x.shape[0], _p(x), _p(norm_w), ctypes.c_float(norm_eps),
                                        _p(x_norm), weights.ref, _p(dout), _p(ids), _p(topw), _p(scores), _p(dx),
                                        ctypes.byref(g), w, n, b, nb, _s(stream)),
            "moe_block_backward")


def moe_layer_forward_host(cfg, x_host, x_dev, weights: Weights, y_dev, y_host, ws, stream=None):
    w, n = _ws(ws)
    N.check(N.load().moe_layer_forward_host(ctypes.byref(cfg), x_host.shape[0], _hp(x_host), _p(x_dev),
                                            weights.ref, _p(y_dev), _hp(y_host), w, n, _s(stream)),
            "moe_layer_forward_host")


def moe_get_device_error(ws, stream=None) -> int:
    code = ctypes.c_int32(0)
    st = N.load().moe_get_device_error(_p(ws), _s(stream), ctypes.byref(code))
    if st not in (N.MOE_OK, N.MOE_ERR_DEVICE):
        N.check(st, "moe_get_device_error")
    return int(code.value)


def moe_clear_device_error(ws, stream=None) -> None:
    N.check(N.load().moe_clear_device_error(_p(ws), _s(stream)), "moe_clear_device_error")


class MoELayer:
    """One layer's config and device weights, with a workspace grown on demand."""

    def __init__(self, cfg: N.MoeConfig, tensors: Dict[str, torch.Tensor]):
        self.cfg = cfg
        self.weights = Weights(tensors)
        self._ws: Optional[torch.Tensor] = None
        self.act = torch.float32 if cfg.act_dtype == N.MOE_DT_F32 else torch.bfloat16

    def enable_sparse_down(self) -> None:
        """Re-lay the expert down weights group-major once, so that decode steps
        skip the 16-neuron groups of W_down whose neurons are all zero."""
        extra = sparse_down_layout(self.cfg, self.weights)
        self.weights = Weights({**self.weights.tensors, **extra})

    def workspace(self, T: int, device) -> torch.Tensor:
        need = workspace_bytes(self.cfg, T)
        if self._ws is None or self._ws.numel() < need or self._ws.device != torch.device(device):
            self._ws = new_workspace(self.cfg, T, device)
        return self._ws

    def forward(self, x: torch.Tensor, y: Optional[torch.Tensor] = None, **outs) -> torch.Tensor:
        if y is None:
            y = torch.empty(x.shape, dtype=self.act, device=x.device)
        moe_layer_forward(self.cfg, x, self.weights, y, self.workspace(x.shape[0], x.device), **outs)
        return y

    __call__ = forward


class MoEBlock(MoELayer):
    """The MoE block of a decoder layer: out = x + layer(RMSNorm(x)), with the
    RMSNorm weight gamma (FP32 [d]) and epsilon; out may be x (in place)."""

    def __init__(self, cfg: N.MoeConfig, tensors: Dict[str, torch.Tensor], norm_w: torch.Tensor,
                 norm_eps: float = 1e-5):
        super().__init__(cfg, tensors)
        self.norm_w = norm_w
        self.norm_eps = float(norm_eps)

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, **outs) -> torch.Tensor:
        if out is None:
            out = torch.empty(x.shape, dtype=self.act, device=x.device)
        moe_block_forward(self.cfg, x, self.norm_w, self.norm_eps, self.weights, out,
                          self.workspace(x.shape[0], x.device), **outs)
        return out

    __call__ = forward
