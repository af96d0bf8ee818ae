"""Seeded synthetic inputs for the routed ReLU^2 MoE layer.

This module draws random numbers and stores them in the layouts the layer
reads; it holds none of the layer's arithmetic.  Both the CUDA path and the
CPU oracle receive the tensors it returns, so the two always see the same
bytes.

Recipe (one generator per tensor, seeded from the workload's ``weight_seed``,
the tensor's id and a replica index):

* hidden rows ``x``               ~ N(0, 1), then stored as the activation dtype;
* every weight matrix             ~ N(0, 1/fan_in) with fan_in = its input width,
                                    stored as BF16 (FP32 for the tiny workload);
* router matrix ``w_router``      ~ N(0, 1/d), FP32, [E, d] (out x in);
* selection bias ``bias``         ~ U(-0.1, 0.1), FP32, plus, for the Zipf
                                    workloads, a fixed per-expert popularity
                                    offset read from ``synth/data``;
* NVFP4 experts                   quantised from the BF16 draws by
                                    round-to-nearest (``quantize_nvfp4``).
* ReLU^2-sparse workloads (``relu_sparsity`` s > 0): trained layers zero most
  expert neurons after ReLU^2, random ones only half.  Every hidden row has
  its component along a seeded unit direction u replaced by a constant c, and
  every expert up row its component along the matching unit direction v of
  the expert input space (v = u, or for latent layers a seeded latent v with
  u = W_ld^T v normalised) replaced by -kappa / 4, with c chosen so that
  v . x_e = 4: a neuron's pre-activation is then about N(-kappa, 1) for every
  row, kappa = Phi^-1(s), and a 16-neuron group of one row is dead with
  probability about s^16.  Replicas of a latent sparse workload share W_ld.
"""
from __future__ import annotations

import os
from typing import Dict, Optional

import numpy as np
import torch

from .configs import BF16, F32, NVFP4, MoEShape

_DATA = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data")

TID_ROUTER, TID_BIAS, TID_LAT_DOWN, TID_LAT_UP, TID_UP, TID_DOWN, TID_SH_UP, TID_SH_DOWN, TID_X, TID_NORM, \
    TID_SPARSE = range(11)
SPARSE_OFFSET = 4.0       # c_e: size of the expert-input offset along v


def _seed(shape: MoEShape, tensor_id: int, replica: int = 0, extra: int = 0) -> int:
    return ((shape.weight_seed * 131 + tensor_id) * 1_000_003 + replica * 7919 + extra) & 0x7FFFFFFFFFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, device, seed: int, dtype: torch.dtype) -> torch.Tensor:
    g = _gen(device, seed)
    out = torch.empty(shape, dtype=dtype, device=device)
    # draw in slabs along the first axis to bound the FP32 temporary
    n0 = shape[0]
    per = max(1, int(2**28 // max(1, int(np.prod(shape[1:])))))
    for i in range(0, n0, per):
        j = min(n0, i + per)
        t = torch.randn((j - i,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        t.mul_(std)
        out[i:j] = t.to(dtype)
    return out


def _act_torch_dtype(code: int) -> torch.dtype:
    return torch.float32 if code == F32 else torch.bfloat16


def zipf_offsets(shape: MoEShape) -> Optional[np.ndarray]:
    """Per-expert popularity offsets added to the selection bias (None if no skew)."""
    if shape.zipf_s == 0.0:
        return None
    path = os.path.join(_DATA, f"zipf_bias_{shape.name}.txt")
    if not os.path.exists(path):
        raise FileNotFoundError(f"popularity offsets for {shape.name} are missing: {path}")
    return np.loadtxt(path, dtype=np.float64).astype(np.float32)


def router_params(shape: MoEShape, with_popularity: bool = True) -> Dict[str, torch.Tensor]:
    """FP32 router matrix [E, d] and selection bias [E], drawn on the CPU."""
    E, d = shape.n_experts, shape.d_model
    w_router = _normal((E, d), d ** -0.5, "cpu", _seed(shape, TID_ROUTER), torch.float32)
    g = _gen("cpu", _seed(shape, TID_BIAS))
    bias = (torch.rand((E,), generator=g, dtype=torch.float32) * 0.2 - 0.1)
    if with_popularity:
        off = zipf_offsets(shape)
        if off is not None:
            bias = bias + torch.from_numpy(off)
    return {"w_router": w_router.contiguous(), "bias": bias.contiguous()}


# ----------------------------------------------------------------------------
# NVFP4 weight encoding (data preparation: turns BF16 draws into stored bytes)
# ----------------------------------------------------------------------------
_E2M1_EDGES_GT = (0.25, 1.25, 2.5, 5.0)     # a value equal to these rounds down (to the even code)
_E2M1_EDGES_GE = (0.75, 1.75, 3.5)          # a value equal to these rounds up (to the even code)


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even onto {0,.5,1,1.5,2,3,4,6}, saturating; returns 4-bit codes."""
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.uint8)
    for e in _E2M1_EDGES_GT:
        code += (a > e).to(torch.uint8)
    for e in _E2M1_EDGES_GE:
        code += (a >= e).to(torch.uint8)
    sign = ((v < 0) & (code > 0)).to(torch.uint8)
    return code | (sign << 3)


def quantize_nvfp4(w: torch.Tensor):
    """Encode one [..., N, K] BF16 tensor per leading index as NVFP4.

    Returns (packed u8 [..., N, K/2], block scales u8 E4M3 [..., N, K/16],
    per-tensor scale f32 [...]).  Encoding: per-tensor scale gs = amax/(6*448);
    block scale sf = E4M3_rn(amax_block / (6*gs)); value code = E2M1_rn(w/(sf*gs)),
    zero where sf is zero; the even K element sits in the low nibble.
    """
    assert w.shape[-1] % 16 == 0
    lead = w.shape[:-2]
    N, K = w.shape[-2], w.shape[-1]
    wf = w.float().reshape(-1, N, K)
    n_t = wf.shape[0]
    q_out = torch.empty((n_t, N, K // 2), dtype=torch.uint8, device=w.device)
    sf_out = torch.empty((n_t, N, K // 16), dtype=torch.uint8, device=w.device)
    gs_out = torch.empty((n_t,), dtype=torch.float32, device=w.device)
    for i in range(n_t):
        t = wf[i]
        amax = t.abs().max()
        gs = (amax / (6.0 * 448.0)).to(torch.float32)
        blk = t.reshape(N, K // 16, 16)
        bmax = blk.abs().amax(dim=-1)
        sf = (bmax / (6.0 * gs)).to(torch.float8_e4m3fn)
        sf_f = sf.to(torch.float32)
        denom = (sf_f * gs).unsqueeze(-1)
        safe = torch.where(denom > 0, denom, torch.ones_like(denom))
        scaled_v = torch.where(denom > 0, blk / safe, torch.zeros_like(blk))
        codes = _e2m1_codes(scaled_v).reshape(N, K)
        q_out[i] = codes[:, 0::2] | (codes[:, 1::2] << 4)
        sf_out[i] = sf.view(torch.uint8)
        gs_out[i] = gs
    return (q_out.reshape(*lead, N, K // 2), sf_out.reshape(*lead, N, K // 16),
            gs_out.reshape(lead) if len(lead) else gs_out.reshape(()))


# ----------------------------------------------------------------------------
def _sparse_frame(shape: MoEShape, device):
    """(u, c, v, kappa) of a ReLU^2-sparse workload: hidden rows get the
    component c along the unit hidden direction u, every expert up row the
    component -kappa / SPARSE_OFFSET along the unit expert-input direction v,
    so that v . x_e = SPARSE_OFFSET for every row.  Latent layers: v is a
    seeded latent direction and u = W_ld^T v normalised (W_ld of replica 0,
    which every replica of a sparse workload shares), c = SPARSE_OFFSET /
    |W_ld^T v|; otherwise u = v, c = SPARSE_OFFSET."""
    from statistics import NormalDist
    g = _gen("cpu", _seed(shape, TID_SPARSE))
    v = torch.randn((shape.d_e,), generator=g, dtype=torch.float32)
    v = v / v.norm()
    if shape.d_latent:
        wld = _normal((shape.d_latent, shape.d_model), shape.d_model ** -0.5, device,
                      _seed(shape, TID_LAT_DOWN, 0), _act_torch_dtype(shape.act_dtype))
        u = wld.float().T @ v.to(device)
        c = SPARSE_OFFSET / float(u.norm())
        u = u / u.norm()
    else:
        u, c = v.to(device), SPARSE_OFFSET
    kappa = NormalDist().inv_cdf(shape.relu_sparsity)
    return u, c, v.to(device), kappa


def _sparsify_up(w_up: torch.Tensor, v: torch.Tensor, kappa: float) -> torch.Tensor:
    """Every up row w -> w - (w . v) v - (kappa / SPARSE_OFFSET) v, expert by expert."""
    v = v.to(w_up.device)
    out = torch.empty_like(w_up)
    for e in range(w_up.shape[0]):
        w = w_up[e].float()
        w = w - (w @ v)[:, None] * v[None, :] - (kappa / SPARSE_OFFSET) * v[None, :]
        out[e] = w.to(w_up.dtype)
    return out


def make_weights(shape: MoEShape, device="cpu", replica: int = 0) -> Dict[str, torch.Tensor]:
    """All weights of one layer.  ``replica`` > 0 draws an independent copy of the
    large tensors (the router and bias are shared by all replicas)."""
    E, d, L, I, S = shape.n_experts, shape.d_model, shape.d_latent, shape.d_expert, shape.d_shared
    de = shape.d_e
    wdt = torch.float32 if shape.expert_dtype == F32 else torch.bfloat16
    sdt = torch.float32 if shape.act_dtype == F32 else torch.bfloat16
    out: Dict[str, torch.Tensor] = {}
    rp = router_params(shape)
    out["w_router"] = rp["w_router"].to(device)
    out["bias"] = rp["bias"].to(device)
    if L:
        # (the ReLU^2-sparse workloads share replica 0's latent down matrix)
        rld = 0 if shape.relu_sparsity > 0 else replica
        out["w_lat_down"] = _normal((L, d), d ** -0.5, device, _seed(shape, TID_LAT_DOWN, rld), sdt)
        out["w_lat_up"] = _normal((d, L), L ** -0.5, device, _seed(shape, TID_LAT_UP, replica), sdt)
    w_up = _normal((E, I, de), de ** -0.5, device, _seed(shape, TID_UP, replica), wdt)
    if shape.relu_sparsity > 0:
        _, _, v, kappa = _sparse_frame(shape, device)
        w_up = _sparsify_up(w_up, v, kappa)
    w_down = _normal((E, de, I), I ** -0.5, device, _seed(shape, TID_DOWN, replica), wdt)
    if shape.expert_dtype == NVFP4:
        out["w_up_q"], out["w_up_sf"], out["w_up_gs"] = quantize_nvfp4(w_up)
        out["w_down_q"], out["w_down_sf"], out["w_down_gs"] = quantize_nvfp4(w_down)
        del w_up, w_down
    else:
        out["w_up"], out["w_down"] = w_up, w_down
    if S:
        out["w_sh_up"] = _normal((S, d), d ** -0.5, device, _seed(shape, TID_SH_UP, replica), sdt)
        out["w_sh_down"] = _normal((d, S), S ** -0.5, device, _seed(shape, TID_SH_DOWN, replica), sdt)
    return out


def make_x(shape: MoEShape, T: int, device="cpu", stream_id: int = 0) -> torch.Tensor:
    """Hidden rows [T, d] ~ N(0,1) in the activation dtype."""
    if T == 0:
        return torch.empty((0, shape.d_model), dtype=_act_torch_dtype(shape.act_dtype), device=device)
    if shape.relu_sparsity > 0:
        # hidden rows with their component along u replaced by c
        z = _normal((T, shape.d_model), 1.0, device, _seed(shape, TID_X, stream_id, extra=T), torch.float32)
        u, c, _, _ = _sparse_frame(shape, device)
        z = z - (z @ u)[:, None] * u[None, :] + c * u[None, :]
        return z.to(_act_torch_dtype(shape.act_dtype))
    return _normal((T, shape.d_model), 1.0, device,
                   _seed(shape, TID_X, stream_id, extra=T), _act_torch_dtype(shape.act_dtype))


def make_norm_weight(shape: MoEShape, device="cpu", replica: int = 0) -> torch.Tensor:
    """RMSNorm weight gamma [d] (FP32) of an MoE block: 1 + U(-0.25, 0.25) per
    column, drawn on the CPU (a weight near one with per-column spread)."""
    g = _gen("cpu", _seed(shape, TID_NORM, replica))
    gamma = 1.0 + (torch.rand((shape.d_model,), generator=g, dtype=torch.float32) * 0.5 - 0.25)
    return gamma.to(device)


def make_calibration_x(shape: MoEShape, T: int) -> torch.Tensor:
    """CPU hidden rows used only to fit the popularity offsets (own seed)."""
    return _normal((T, shape.d_model), 1.0, "cpu", _seed(shape, TID_X, 4242), _act_torch_dtype(shape.act_dtype))


def zipf_targets(E: int, K: int, s: float, seed: int) -> np.ndarray:
    """Per-expert pick rates f_e with f_rank = min(1, c * rank^-s) and sum f = K.

    Ranks come from a seeded permutation so popularity is not tied to low ids
    or to one group.  (Distribution shaping only; no routing arithmetic.)"""
    r = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    lo, hi = 0.0, 1e6
    for _ in range(200):
        c = 0.5 * (lo + hi)
        if np.minimum(1.0, c * r).sum() > K:
            hi = c
        else:
            lo = c
    f_rank = np.minimum(1.0, lo * r)
    perm = np.random.default_rng([seed, 7]).permutation(E)
    f = np.empty(E)
    f[perm] = f_rank            # expert perm[i] has rank i+1
    return f
