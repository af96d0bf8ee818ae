"""Shared helpers of the GPU parity tests: run the CUDA library on seeded inputs
and evaluate the oracle on the same bytes."""
from __future__ import annotations

import functools
from typing import Dict, Optional

import numpy as np
import torch

from oracle import moe_oracle as O
from synth import BF16, F32, MoEShape, make_weights, make_x

import routed_relu_expert_gb300 as M

# tolerances (max |y - y_ref| / RMS(y_ref)); the BF16 and NVFP4 bars are the
# layer's stated contract, the FP32 one is a tighter reading for FP32 layers
TOL_BF16 = 2e-2
TOL_NVFP4 = 5e-2
TOL_F32 = 1e-4
TOL_W = 1e-6          # routing weights, absolute
TOL_LOGIT = 1e-5      # logits, relative to sum_i |x_i W_ei|


@functools.lru_cache(maxsize=4)
def device_weights(shape: MoEShape, replica: int = 0) -> Dict[str, torch.Tensor]:
    return make_weights(shape, "cuda", replica)


class _ExpertRows:
    """weights["w_up"][e] -> float64 numpy of one expert, copied on demand."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].float().cpu().numpy().astype(np.float64)


def oracle_weights(w: Dict[str, torch.Tensor]) -> Dict[str, object]:
    out = {}
    for k, v in w.items():
        if k in ("w_up", "w_down", "w_up_q", "w_down_q", "w_up_sf", "w_down_sf"):
            out[k] = _ExpertRows(v) if v.dtype != torch.uint8 else _U8Rows(v)
        elif k in ("w_router", "bias"):
            out[k] = v.cpu().numpy()
        elif k in ("w_up_gs", "w_down_gs"):
            out[k] = v.cpu().numpy().astype(np.float64)
        else:
            out[k] = v.float().cpu().numpy().astype(np.float64)
    return out


class _U8Rows:
    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].cpu().numpy()


def run_gpu(shape: MoEShape, w: Dict[str, torch.Tensor], x: torch.Tensor):
    cfg = M.config_from(shape)
    T = x.shape[0]
    E, K = shape.n_experts, shape.top_k
    layer = M.MoELayer(cfg, w)
    y = torch.empty_like(x)
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    topw = torch.empty((T, K), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    scores = torch.empty((T, E), dtype=torch.float32, device="cuda")
    layer.forward(x, y, ids_out=ids, topw_out=topw, logits_out=logits, scores_out=scores)
    ws = layer.workspace(T, x.device)
    err = M.moe_get_device_error(ws)
    torch.cuda.synchronize()
    return {"y": y, "ids": ids, "topw": topw, "logits": logits, "scores": scores, "err": err, "layer": layer,
            "ws": ws}


def ws_table(ws: torch.Tensor, cfg, T: int, region: int, dtype: torch.dtype) -> torch.Tensor:
    """A route table (or row region) the layer left in its workspace, as a flat
    device tensor view."""
    off, nbytes = M.workspace_region(cfg, T, region)
    return ws[off:off + nbytes].view(dtype)


def check_route_tables(shape: MoEShape, ws: torch.Tensor, ids_gpu: np.ndarray, T: int) -> Dict[str, np.ndarray]:
    """The dispatch tables moe_layer_forward left in its workspace (counts,
    offsets, per-expert token lists, slots, inverse map) bit-exact against the
    oracle's dispatch of the same expert ids.  Returns the oracle's tables."""
    from routed_relu_expert_gb300 import _native as N
    cfg = M.config_from(shape)
    ref = O.dispatch(ids_gpu, shape.n_experts)
    for region, key in ((N.MOE_WS_COUNTS, "counts"), (N.MOE_WS_OFFSETS, "offsets"),
                        (N.MOE_WS_ROUTE_TOKEN, "route_token"), (N.MOE_WS_ROUTE_SLOT, "route_slot"),
                        (N.MOE_WS_TOKEN_SLOT_ROW, "token_slot_row")):
        got = ws_table(ws, cfg, T, region, torch.int32).cpu().numpy().astype(np.int64)
        assert np.array_equal(got, ref[key].reshape(-1)), f"{key} differs from the oracle's dispatch"
    return ref


def check_router(shape: MoEShape, x_np: np.ndarray, ow: Dict, g: Dict, rows: Optional[np.ndarray] = None):
    """Router checks on GPU outputs g (numpy): logits vs FP64, scores within
    4 ulp of the sigmoid of the GPU's own logits, ids bit-exact and weights
    1e-6 vs the oracle's selection on the GPU's scores.  Returns the oracle's
    (ids, w)."""
    rows = np.arange(x_np.shape[0]) if rows is None else rows
    z, zs = O.router_logits(x_np[rows], ow["w_router"])
    lg = g["logits"][rows].astype(np.float64)
    assert np.all(np.abs(lg - z) <= TOL_LOGIT * zs), f"logit error {np.max(np.abs(lg - z) / zs)}"
    s_ref = O.sigmoid_scores(g["logits"][rows])
    ulp = np.abs(g["scores"][rows].view(np.int32).astype(np.int64) - s_ref.view(np.int32).astype(np.int64))
    # CUDA's expf is within 2 ulp; 1 + e and the division add one rounding each
    assert ulp.max() <= 4, f"sigmoid differs by {ulp.max()} ulp"
    ids_o, w_o = O.route(g["scores"][rows], ow.get("bias"), shape.n_group, shape.topk_group, shape.top_k,
                         shape.norm_topk_prob, shape.routed_scaling_factor)
    mism = np.where(np.any(ids_o != g["ids"][rows], axis=1))[0]
    assert mism.size == 0, f"{mism.size} tokens routed differently, first {rows[mism[:5]]}"
    assert np.max(np.abs(w_o - g["topw"][rows].astype(np.float64))) <= TOL_W
    return ids_o, w_o


def check_output(shape: MoEShape, x_np: np.ndarray, ow: Dict, ids_o, w_o, y_gpu: np.ndarray, tol: float,
                 rows: Optional[np.ndarray] = None, chunk: int = 0) -> float:
    """max |y - y_ref| / RMS(y_ref) over the given rows (all by default), the
    oracle evaluated on the GPU's routing; ``chunk`` > 0 evaluates the oracle
    that many rows at a time (the layer is per token, so the result is the
    same; only host memory is bounded)."""
    rows = np.arange(x_np.shape[0]) if rows is None else rows
    ids_o, w_o = np.asarray(ids_o), np.asarray(w_o)
    step = chunk if chunk > 0 else len(rows)
    worst, sq, n = 0.0, 0.0, 0
    for i in range(0, len(rows), step):
        sel = rows[i:i + step]
        ref = O.layer_forward(x_np[sel], ow, ids_o[i:i + step], w_o[i:i + step], shape.n_experts,
                              bf16_points=shape.act_dtype == BF16)["y"]
        worst = max(worst, float(np.max(np.abs(y_gpu[sel].astype(np.float64) - ref))))
        sq += float(np.sum(ref ** 2))
        n += ref.size
    rms = (sq / n) ** 0.5
    err = worst / rms
    assert err <= tol, f"max |y - y_ref| = {err:.3e} RMS > {tol}"
    return err


def to_np(g):
    out = {}
    for k, v in g.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy()
        else:
            out[k] = v
    return out


def tol_of(shape: MoEShape) -> float:
    if shape.act_dtype == F32:
        return TOL_F32
    return TOL_NVFP4 if shape.expert_dtype == 2 else TOL_BF16
