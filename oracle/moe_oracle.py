"""CPU oracle for the routed ReLU^2 mixture-of-experts feed-forward layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may load it.  It shares no code, table or helper with the CUDA
library.

It is the layer written out as its definition, slowly and plainly, in NumPy
float64, with the two kinds of precision the pages fix:

* the router works on FP32 logits and FP32 sigmoid scores, the selection bias
  enters only the choice, ties go to the lower expert id
  (page "NemotronH (Nemotron 3.5 Lightning, Bolt, Super VL)", section
  "Arithmetic", router bullet; page "Nemotron Is Not One Circuit", section
  "The Router Is A Deterministic Algorithm");
* an expert rounds to BF16 after its up projection and again after the
  squared ReLU, ``bf16(relu(bf16(up x))^2)``, then applies its down
  projection; routed outputs are summed per token in ascending expert id
  (page "NemotronH ...", section "Arithmetic", experts bullet).

Everything else is float64.  The layer output is returned *before* its final
storage rounding to BF16, so a comparison charges the device's own storage
rounding (at most half a BF16 unit in the last place) to the device.

Readings taken where the pages are silent (each is listed in the design notes):
router input is the hidden row (not the latent row); groups are equal
contiguous id ranges and a tie in group score goes to the lower group index;
experts outside the kept groups cannot be chosen; the chosen ids are listed in
descending biased score; normalisation has no epsilon; the shared expert is
added without a gate; for latent layers the latent down output is rounded to
BF16 (the experts' input dtype), the combined latent vector is rounded once
to BF16 before the latent up projection, and the latent up output is added
to the shared expert's output.

Parity pins for every function here live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import math
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------


def bf16_round(a) -> np.ndarray:
    """Round float64 values to the nearest BF16 value, ties to even (one rounding).

    BF16 keeps 8 significant bits and FP32's exponent range; values are
    returned as float64.  Written from the format's definition: split
    a = m * 2^e with m in [0.5, 1), keep round_half_even(m * 2^8) / 2^8,
    with the quantum fixed at 2^-133 below the smallest normal (2^-126)."""
    a = np.asarray(a, dtype=np.float64)
    out = a.copy()
    fin = np.isfinite(a) & (a != 0)
    m, e = np.frexp(a[fin])                    # a = m * 2^e, 0.5 <= |m| < 1
    # exponent of the leading bit is e-1; quantum = 2^(e-1-7), floored at 2^-133
    q_exp = np.maximum(e - 8, -133)
    q = np.ldexp(np.ones_like(m), q_exp)
    r = np.rint(a[fin] / q) * q                # np.rint rounds half to even
    r[np.abs(r) >= 2.0 ** 128] = np.inf * np.sign(r[np.abs(r) >= 2.0 ** 128])
    out[fin] = r
    return out


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (sign, 2 exponent bits, 1 mantissa bit, bias 1).

    NVFP4 element format: subnormal when the exponent field is zero."""
    s = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * 0.5 * m
    return s * (2.0 ** (e - 1)) * (1.0 + 0.5 * m)


def e4m3_value(byte: int) -> float:
    """Value of an 8-bit E4M3 code (sign, 4 exponent bits bias 7, 3 mantissa bits).

    No infinities; exponent field 15 with mantissa 7 is NaN; largest value 448."""
    s = -1.0 if (byte >> 7) & 1 else 1.0
    E = (byte >> 3) & 15
    M = byte & 7
    if E == 15 and M == 7:
        return float("nan")
    if E == 0:
        return s * (M / 8.0) * 2.0 ** -6
    return s * (2.0 ** (E - 7)) * (1.0 + M / 8.0)


_E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def dequant_nvfp4(q: np.ndarray, sf: np.ndarray, gs) -> np.ndarray:
    """NVFP4 -> float64: value = E2M1(nibble) * E4M3(block scale) * per-tensor scale.

    ``q`` [..., N, K/2] u8 with element 2j in the low nibble and 2j+1 in the
    high nibble; ``sf`` [..., N, K/16] u8, one scale per 16 consecutive K
    elements ("Nemotron-3.5-Super 120B on an 8 GB GPU", section "The engine,
    step by step", item 4); ``gs`` scalar or [...] f32 per tensor."""
    q = np.asarray(q, dtype=np.uint8)
    lo = _E2M1_TABLE[q & 0xF]
    hi = _E2M1_TABLE[q >> 4]
    vals = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.float64)
    vals[..., 0::2] = lo
    vals[..., 1::2] = hi
    scale = _E4M3_TABLE[np.asarray(sf, dtype=np.uint8)]
    vals = vals * np.repeat(scale, 16, axis=-1)
    gs = np.asarray(gs, dtype=np.float64)
    return vals * gs.reshape(gs.shape + (1, 1))


# ----------------------------------------------------------------------------
# NVFP4 activation terms (the FP4 tensor-core path).  The NVFP4 block format
# -- E2M1 values, one E4M3 scale per 16 consecutive values, one FP32 scale
# per tensor -- is the one of page "Nemotron-3.5-Super 120B on an 8 GB GPU",
# section "The engine, step by step", item 4.  A row of activations is split
# into n terms of that format, each quantising what the previous terms left
# (residual quantisation), so the products can run with both operands in
# NVFP4; n = 1 is plain W4A4.  Every decision is taken in FP32, as the device
# takes it: g = amax(row) / (6 * 448); per term and 16-value block,
# scale = E4M3_rn(amax(block) / (6 g)) (saturating), s = scale * g,
# code = E2M1_rn(r * (1 / s)) (saturating; 0 where s = 0), r -= code * s.
# ----------------------------------------------------------------------------
_E2M1_GRID = np.array([e2m1_value(c) for c in range(8)], dtype=np.float64)          # codes 0..7
_E4M3_GRID = np.array([e4m3_value(b) for b in range(127)], dtype=np.float64)        # codes 0..126 (127 = NaN)


def _rne_code(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Code of the nearest value of an increasing grid to a >= 0, ties to the
    even code, values beyond the last one saturating to it."""
    a = np.minimum(np.asarray(a, dtype=np.float64), grid[-1])
    hi = np.clip(np.searchsorted(grid, a, side="left"), 0, len(grid) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - grid[lo], grid[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(a == grid[hi], hi, np.where(take_hi, hi, lo)).astype(np.uint8)


def e4m3_rn_code(v) -> np.ndarray:
    """E4M3 code of the nearest E4M3 value to v >= 0 (ties to even, saturating at 448)."""
    return _rne_code(v, _E4M3_GRID)


def e2m1_rn_code(v) -> np.ndarray:
    """Signed 4-bit E2M1 code of the nearest E2M1 value to v (ties to even,
    saturating at +-6); a value that rounds to zero gets the code 0."""
    v = np.asarray(v, dtype=np.float64)
    c = _rne_code(np.abs(v), _E2M1_GRID)
    return np.where((v < 0) & (c > 0), c | 8, c).astype(np.uint8)


def nvfp4_terms(x: np.ndarray, n_terms: int):
    """Rows x [T, K] (FP32 values; K a multiple of 16) -> (codes [n, T, K] u8
    signed E2M1 codes, scales [n, T, K/16] u8 E4M3 codes, g [T] FP32)."""
    x = np.asarray(x, dtype=np.float32)
    T, K = x.shape
    g = (np.max(np.abs(x), axis=1) / np.float32(6.0 * 448.0)).astype(np.float32) if K else np.zeros(T, np.float32)
    g = np.where(g > 0, g, np.float32(1.0)).astype(np.float32)
    six_g = (np.float32(6.0) * g).astype(np.float32)
    r = x.reshape(T, K // 16, 16).copy()
    codes = np.zeros((n_terms, T, K // 16, 16), dtype=np.uint8)
    scales = np.zeros((n_terms, T, K // 16), dtype=np.uint8)
    for j in range(n_terms):
        amax_b = np.max(np.abs(r), axis=2).astype(np.float32)
        sf = e4m3_rn_code((amax_b / six_g[:, None]).astype(np.float32))
        s = (_E4M3_GRID[sf].astype(np.float32) * g[:, None]).astype(np.float32)
        inv = np.where(s > 0, np.float32(1) / np.where(s > 0, s, np.float32(1)), np.float32(0)).astype(np.float32)
        ratio = (r * inv[..., None]).astype(np.float32)
        c = e2m1_rn_code(ratio.astype(np.float32))
        q = (np.where(c & 8, -1.0, 1.0) * _E2M1_GRID[c & 7]).astype(np.float32)
        r = (r - (q * s[..., None]).astype(np.float32)).astype(np.float32)
        codes[j], scales[j] = c, sf
    return codes.reshape(n_terms, T, K), scales, g


def dequant_terms(codes: np.ndarray, scales: np.ndarray, g: np.ndarray) -> np.ndarray:
    """Sum over terms of E2M1(code) * E4M3(scale) * g, float64 [T, K]."""
    n, T, K = codes.shape
    v = np.where(codes & 8, -1.0, 1.0) * _E2M1_GRID[codes & 7]
    v = v.reshape(n, T, K // 16, 16) * _E4M3_TABLE[scales][..., None]
    return v.sum(axis=0).reshape(T, K) * np.asarray(g, dtype=np.float64)[:, None]


def nvfp4_activations(x: np.ndarray, n_terms: int) -> np.ndarray:
    """x replaced by the sum of its n_terms NVFP4 terms (float64)."""
    return dequant_terms(*nvfp4_terms(x, n_terms))


# ----------------------------------------------------------------------------
# router (page "Nemotron Is Not One Circuit", "The Router Is A Deterministic
# Algorithm" and "The C Kernel Contract")
# ----------------------------------------------------------------------------


def router_logits(x: np.ndarray, w_router: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Router projection Z = X W_r^T with the stored [E, d] matrix
    (page "M6.1 Routed Capacity", section 0x04A).  Returns (z, scale) where
    scale[t, e] = sum_i |x_ti W_ei| bounds the rounding error of any
    summation order (used for the relative logit check)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    return x @ w.T, np.abs(x) @ np.abs(w).T


def sigmoid_scores(z) -> np.ndarray:
    """FP32 sigmoid scores s = 1/(1+exp(-z)) of FP32 logits, correctly rounded
    to FP32 from a float64 evaluation."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-z))
    return s.astype(np.float32)


def _rank_desc(values: np.ndarray, index: np.ndarray) -> np.ndarray:
    """Order of ``index`` by value descending, equal values by lower index,
    NaN after everything else."""
    v = np.asarray(values, dtype=np.float64)
    key = np.where(np.isnan(v), np.inf, -v)
    index = np.asarray(index, dtype=np.int64)
    return index[np.lexsort((index, key))]      # primary: key, secondary: index


def select_token(scores: np.ndarray, bias: Optional[np.ndarray], n_group: int,
                 topk_group: int, top_k: int) -> np.ndarray:
    """Group-limited top-k of one token.

    Biased score c = s + b in FP32 (bias affects only the choice).  Experts are
    cut into n_group equal contiguous groups; a group's score is the FP32 sum of
    its two largest c; the topk_group best groups survive (ties: lower group);
    the top_k experts by c among the survivors are returned in descending c,
    equal c to the lower id."""
    s = np.asarray(scores, dtype=np.float32)
    E = s.shape[0]
    c = s + (np.asarray(bias, dtype=np.float32) if bias is not None else np.float32(0))
    c = c.astype(np.float32)
    if n_group > 1 and topk_group < n_group:
        gsz = E // n_group
        gscore = np.empty(n_group, dtype=np.float32)
        for g in range(n_group):
            grp = c[g * gsz:(g + 1) * gsz]
            top2 = _rank_desc(grp, np.arange(gsz))[:2]
            gscore[g] = np.float32(grp[top2[0]]) + np.float32(grp[top2[1]])
        kept = sorted(_rank_desc(gscore, np.arange(n_group))[:topk_group].tolist())
        cand = np.concatenate([np.arange(g * gsz, (g + 1) * gsz) for g in kept])
    else:
        cand = np.arange(E)
    return _rank_desc(c[cand], cand)[:top_k]


def select_batch(scores: np.ndarray, bias: Optional[np.ndarray], n_group: int,
                 topk_group: int, top_k: int) -> np.ndarray:
    """``select_token`` for every row at once (same rule, same FP32 sums), used
    where many tokens are routed; pinned against ``select_token`` in the tests."""
    s = np.asarray(scores, dtype=np.float32)
    T, E = s.shape
    c = (s + (np.asarray(bias, dtype=np.float32) if bias is not None else np.float32(0))).astype(np.float32)
    idx = np.broadcast_to(np.arange(E), (T, E))
    kept = np.ones((T, E), dtype=bool)
    if n_group > 1 and topk_group < n_group:
        gsz = E // n_group
        cg = np.where(np.isnan(c), -np.inf, c).reshape(T, n_group, gsz)
        top2 = np.sort(cg, axis=-1)[..., -2:]
        gscore = (top2[..., 1] + top2[..., 0]).astype(np.float32)
        gidx = np.broadcast_to(np.arange(n_group), (T, n_group))
        gorder = np.lexsort((gidx, -gscore.astype(np.float64)), axis=-1)[:, :topk_group]
        gkeep = np.zeros((T, n_group), dtype=bool)
        np.put_along_axis(gkeep, gorder, True, axis=-1)
        kept = np.repeat(gkeep, gsz, axis=-1)
    cd = c.astype(np.float64)
    key = np.where(np.isnan(cd), np.inf, -cd)
    order = np.lexsort((idx, key, ~kept), axis=-1)
    return order[:, :top_k].astype(np.int64)


def routing_weights(scores: np.ndarray, ids: np.ndarray, norm_topk_prob: int,
                    routed_scaling_factor: float) -> np.ndarray:
    """Weights gathered from the *unbiased* scores of the chosen experts,
    normalised to sum one if configured, then times the routed scaling factor."""
    w = np.asarray(scores, dtype=np.float64)[np.asarray(ids)]
    if norm_topk_prob:
        w = w / w.sum()
    return w * float(routed_scaling_factor)


def route(scores: np.ndarray, bias: Optional[np.ndarray], n_group: int, topk_group: int,
          top_k: int, norm_topk_prob: int, rsf: float) -> Tuple[np.ndarray, np.ndarray]:
    """Selection and weights for every token: scores [T, E] f32 -> ids [T, K] i32, w [T, K] f64."""
    scores = np.asarray(scores, dtype=np.float32)
    T = scores.shape[0]
    ids = np.zeros((T, top_k), dtype=np.int32)
    w = np.zeros((T, top_k), dtype=np.float64)
    for t in range(T):
        ids[t] = select_token(scores[t], bias, n_group, topk_group, top_k)
        w[t] = routing_weights(scores[t], ids[t], norm_topk_prob, rsf)
    return ids, w


def boundary_margin(scores: np.ndarray, bias: Optional[np.ndarray], ids: np.ndarray) -> np.ndarray:
    """Per token: biased score of the last chosen expert minus the best biased
    score left out (page "M6.1 Routed Capacity", section 0x04D, top-k boundary
    margin).  Small margins flag tokens whose choice a one-ulp change can flip.
    This is the plain top-k margin over all experts: under group limits a
    negative value means a dropped group held a higher score."""
    s = np.asarray(scores, dtype=np.float32)
    c = (s + (np.asarray(bias, dtype=np.float32) if bias is not None else np.float32(0))).astype(np.float64)
    T, E = c.shape
    out = np.empty(T)
    for t in range(T):
        chosen = np.zeros(E, dtype=bool)
        chosen[ids[t]] = True
        rest = c[t][~chosen]
        out[t] = c[t][ids[t][-1]] - (rest.max() if rest.size else -np.inf)
    return out


# ----------------------------------------------------------------------------
# dispatch and combine (page "M6.1 Routed Capacity", sections 0x05A-0x05E)
# ----------------------------------------------------------------------------


def dispatch(ids: np.ndarray, n_experts: int) -> Dict[str, np.ndarray]:
    """Expert-contiguous route layout.

    Routes (token t, slot k, expert ids[t,k]) are sorted by (expert, token, slot);
    offsets are the exclusive prefix sum of per-expert counts (E+1 entries);
    token_slot_row[t, k] is the packed row of route (t, k)."""
    ids = np.asarray(ids, dtype=np.int64)
    T, K = ids.shape
    tok = np.repeat(np.arange(T), K)
    slot = np.tile(np.arange(K), T)
    exp = ids.reshape(-1)
    order = np.lexsort((slot, tok, exp))          # primary key: expert, then token, then slot
    counts = np.bincount(exp, minlength=n_experts).astype(np.int64)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    route_token = tok[order]
    route_slot = slot[order]
    token_slot_row = np.empty((T, K), dtype=np.int64)
    token_slot_row[route_token, route_slot] = np.arange(T * K)
    return {"counts": counts, "offsets": offsets, "route_token": route_token,
            "route_slot": route_slot, "token_slot_row": token_slot_row,
            "route_expert": exp[order]}


def moe_apply(h: np.ndarray, ids: np.ndarray, gates: np.ndarray,
              experts: Sequence[Callable[[np.ndarray], np.ndarray]]) -> np.ndarray:
    """Packed gather -> per-expert evaluation -> weighted scatter-add.

    X_packed[j] = H[a_pi(j)];  Y_t = sum over packed rows j of token t of
    g_pi(j) U_j, summed in packed (ascending expert) order."""
    h = np.asarray(h, dtype=np.float64)
    T = h.shape[0]
    meta = dispatch(ids, len(experts))
    x_packed = h[meta["route_token"]]
    g = np.asarray(gates, dtype=np.float64)[meta["route_token"], meta["route_slot"]]
    off = meta["offsets"]
    y = None
    for e in range(len(experts)):
        lo, hi = int(off[e]), int(off[e + 1])
        if lo == hi:
            continue
        u = np.asarray(experts[e](x_packed[lo:hi]), dtype=np.float64)
        if y is None:
            y = np.zeros((T, u.shape[1]), dtype=np.float64)
        for j in range(lo, hi):
            y[meta["route_token"][j]] += g[j] * u[j - lo]
    if y is None:
        y = np.zeros((T, h.shape[1]), dtype=np.float64)
    return y


# ----------------------------------------------------------------------------
# experts
# ----------------------------------------------------------------------------


def relu2_mlp(x: np.ndarray, w_up: np.ndarray, w_down: np.ndarray, bf16_points: bool,
              act_terms: Optional[int] = None) -> np.ndarray:
    """ReLU^2 MLP without gate: W_down relu(W_up x)^2 with stored [out, in]
    matrices; with ``bf16_points`` the up output and the squared ReLU are each
    rounded to BF16 (page "NemotronH ...", section "Arithmetic").  With
    ``act_terms`` the inputs of both products (x and h) are replaced by their
    NVFP4 terms (``nvfp4_activations``)."""
    x = np.asarray(x, dtype=np.float64)
    if act_terms:
        x = nvfp4_activations(x, act_terms)
    a = x @ np.asarray(w_up, dtype=np.float64).T
    if bf16_points:
        a = bf16_round(a)
    h = np.maximum(a, 0.0) ** 2
    if bf16_points:
        h = bf16_round(h)
    if act_terms:
        h = nvfp4_activations(h, act_terms)
    return h @ np.asarray(w_down, dtype=np.float64).T


def expert_matrices(weights: Dict[str, np.ndarray], e: int) -> Tuple[np.ndarray, np.ndarray]:
    """(W_up [I, de], W_down [de, I]) of expert e as float64 (NVFP4 dequantised)."""
    if "w_up_q" in weights:
        up = dequant_nvfp4(weights["w_up_q"][e], weights["w_up_sf"][e], weights["w_up_gs"][e])
        down = dequant_nvfp4(weights["w_down_q"][e], weights["w_down_sf"][e], weights["w_down_gs"][e])
        return up, down
    return (np.asarray(weights["w_up"][e], dtype=np.float64),
            np.asarray(weights["w_down"][e], dtype=np.float64))


def layer_forward(x: np.ndarray, weights: Dict[str, np.ndarray], ids: np.ndarray, w: np.ndarray,
                  n_experts: int, bf16_points: bool, act_terms: Optional[int] = None) -> Dict[str, np.ndarray]:
    """MoE layer output for given routing (ids [T,K], weights w [T,K]).

    Steps: latent down (if any) -> packed dispatch -> per expert ReLU^2 MLP ->
    weighted scatter-add in ascending expert id -> shared expert -> latent up
    (if any) -> sum.  No residual and no norm (page "M6.1 Routed Capacity",
    section 0x05F: the residual is not part of the MoE output).  Returns the
    float64 output before storage rounding plus the intermediates.
    ``act_terms``: the routed experts' input rows and h enter their products
    as NVFP4 terms (``relu2_mlp``); the shared expert is unchanged."""
    x = np.asarray(x, dtype=np.float64)
    latent = "w_lat_down" in weights
    if latent:
        x_e = x @ np.asarray(weights["w_lat_down"], dtype=np.float64).T
        if bf16_points:
            x_e = bf16_round(x_e)
    else:
        x_e = x
    experts = []
    for e in range(n_experts):
        experts.append(_LazyExpert(weights, e, bf16_points, act_terms))
    y_r = moe_apply(x_e, ids, w, experts)
    out = {"y_routed": y_r, "x_e": x_e}
    if "w_sh_up" in weights:
        y_s = relu2_mlp(x, weights["w_sh_up"], weights["w_sh_down"], bf16_points)
    else:
        y_s = np.zeros((x.shape[0], x.shape[1]), dtype=np.float64)
    out["y_shared"] = y_s
    if latent:
        y_lat = bf16_round(y_r) if bf16_points else y_r
        y = y_lat @ np.asarray(weights["w_lat_up"], dtype=np.float64).T + y_s
    else:
        y = y_r + y_s
    out["y"] = y
    return out


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of every row, float64: gamma * x / sqrt(mean(x^2) + eps)
    (page "Nemotron Is Not One Circuit", section "The Four Layer Kinds CKE Must
    Preserve": an MoE layer starts with RMSNorm).  The pages name the step
    only; this is its usual definition, a root mean square over the hidden
    width, no mean subtraction, a learned per-column weight."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=1, keepdims=True)
    return np.asarray(gamma, dtype=np.float64)[None, :] * (x / np.sqrt(ms + eps))


def block_forward(x: np.ndarray, gamma: np.ndarray, eps: float, weights: Dict[str, np.ndarray],
                  ids: np.ndarray, w: np.ndarray, n_experts: int, bf16_points: bool,
                  xn: Optional[np.ndarray] = None, act_terms: Optional[int] = None) -> Dict[str, np.ndarray]:
    """MoE block of a decoder layer for given routing: out = x + layer(RMSNorm(x))
    (page "Nemotron Is Not One Circuit", section "The Four Layer Kinds CKE Must
    Preserve": RMSNorm -> router -> group-limited top-k -> routed ReLU^2 experts
    + shared expert -> residual).  ``xn``: the normalised rows the layer reads,
    when they are given as the device stored them (rounded to its activation
    type); else the float64 ``rms_norm``.  Returns the float64 ``out`` before
    storage rounding, ``xn`` and the layer's intermediates."""
    xn_ref = rms_norm(x, gamma, eps)
    xl = xn_ref if xn is None else np.asarray(xn, dtype=np.float64)
    out = layer_forward(xl, weights, ids, w, n_experts, bf16_points, act_terms)
    out["xn_ref"] = xn_ref
    out["out"] = np.asarray(x, dtype=np.float64) + out["y"]
    return out


# ----------------------------------------------------------------------------
# backward (page "M6.1 Routed Capacity", section 0x06F: the forward relation is
# frozen, the route tensors are the coordinates of the backward; combine
# backward is a broadcast and a dot product, the gather's adjoint a
# scatter-add, and the router and expert paths meet again at the input)
# ----------------------------------------------------------------------------


def gate_backward(scores_sel: np.ndarray, q: np.ndarray, norm_topk_prob: int, rsf: float) -> np.ndarray:
    """dL/ds of the chosen experts' scores from q = dL/dw.  The weights are
    w_k = rsf s_k / sum_j s_j (or rsf s_k without normalisation), so
    dL/ds_j = rsf / S (q_j - sum_k q_k s_k / S), S = sum_j s_j.  This is the
    page's selected-gate Jacobian contraction (section 0x06F.3) for this
    layer's sigmoid-then-normalise gate instead of a selected softmax."""
    s = np.asarray(scores_sel, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    if not norm_topk_prob:
        return rsf * q
    S = s.sum(axis=-1, keepdims=True)
    return rsf / S * (q - (q * s).sum(axis=-1, keepdims=True) / S)


def layer_backward(x: np.ndarray, weights: Dict[str, np.ndarray], ids: np.ndarray, scores: np.ndarray,
                   dy: np.ndarray, n_experts: int, norm_topk_prob: int, rsf: float,
                   bf16_points: bool = False) -> Dict[str, object]:
    """Gradients of L = <dy, y> for the layer with its routing frozen.

    The chosen ids are fixed metadata (no gradient; the selection bias only
    chooses); ``scores`` [T, E] are the forward's sigmoid scores.  Real
    arithmetic in float64: no rounding point of the forward is modelled.
    Per route r = (t, k) of expert e (page section 0x06F.2, 0x06F.6):
      U_r = W_down,e relu(a_r)^2, a_r = W_up,e x_e,t;   q_r = <dy_r,t, U_r>;
      dU_r = w_r dy_r,t;  dh_r = W_down,e^T dU_r;  da_r = dh_r * 2 relu(a_r);
      dW_down,e += dU_r h_r^T;  dW_up,e += da_r x_e,t^T;  dx_e,t += W_up,e^T da_r
    (dy_r = dy, or dy W_lu for latent layers, where dW_lu = dy^T y_r).
    ``bf16_points``: the forward's rounding points (latent rows, a, h, the
    latent combine y_r; see ``relu2_mlp``) and a BF16 reading of the
    backward's tensor-core operands: dy_r = bf16(dy W_lu), dU = bf16(w dy_r),
    da = bf16(dh * 2 sqrt(h)) (relu(a) taken from the stored h), the latent
    input gradient rounded before its two products, and the shared expert's
    da_s = bf16((dy W_sd) * 2 sqrt(h_s)); everything else stays float64.
    Gates (section 0x06F.3, 0x06F.4): ds from q (``gate_backward``),
    dz = ds s (1 - s) at the chosen experts, zero elsewhere;
    dW_r += dz x_t per chosen expert, dx_t += dz W_r,e.
    Shared expert: the dense ReLU^2 MLP's backward on x.  Latent down:
    dW_ld = dx_e^T x, dx += dx_e W_ld; otherwise dx += dx_e."""
    x = np.asarray(x, dtype=np.float64)
    D = np.asarray(dy, dtype=np.float64)
    ids = np.asarray(ids)
    T, K = ids.shape
    s_all = np.asarray(scores, dtype=np.float64)
    s_sel = np.take_along_axis(s_all, ids.astype(np.int64), axis=1)
    w = rsf * (s_sel / s_sel.sum(axis=1, keepdims=True) if norm_topk_prob else s_sel)
    latent = "w_lat_down" in weights
    out: Dict[str, object] = {}
    dx = np.zeros_like(x)
    rnd = bf16_round if bf16_points else (lambda v: v)
    if latent:
        W_ld = np.asarray(weights["w_lat_down"], dtype=np.float64)
        x_e = rnd(x @ W_ld.T)
    else:
        x_e = x
    de = x_e.shape[1]
    # routed experts, route by route
    y_r = np.zeros((T, de))
    U = np.zeros((T, K, de))
    acts = {}
    for t in range(T):
        for k in range(K):
            e = int(ids[t, k])
            up, down = expert_matrices(weights, e)
            a = rnd(up @ x_e[t])
            h = rnd(np.maximum(a, 0.0) ** 2)
            U[t, k] = down @ h
            acts[(t, k)] = (a, h)
            y_r[t] += w[t, k] * U[t, k]
    if latent:
        W_lu = np.asarray(weights["w_lat_up"], dtype=np.float64)
        dy_r = rnd(D @ W_lu)
        out["d_w_lat_up"] = D.T @ rnd(y_r)
    else:
        dy_r = D
    q = np.einsum("td,tkd->tk", dy_r, U)
    d_up: Dict[int, np.ndarray] = {}
    d_down: Dict[int, np.ndarray] = {}
    dx_e = np.zeros_like(x_e)
    for t in range(T):
        for k in range(K):
            e = int(ids[t, k])
            up, down = expert_matrices(weights, e)
            a, h = acts[(t, k)]
            dU = rnd(w[t, k] * dy_r[t])
            dh = down.T @ dU
            da = rnd(dh * 2.0 * np.sqrt(h)) if bf16_points else dh * 2.0 * np.maximum(a, 0.0)
            d_down[e] = d_down.get(e, 0.0) + np.outer(dU, h)
            d_up[e] = d_up.get(e, 0.0) + np.outer(da, x_e[t])
            dx_e[t] += up.T @ da
    ds = gate_backward(s_sel, q, norm_topk_prob, rsf)
    dz = ds * s_sel * (1.0 - s_sel)
    W_r = np.asarray(weights["w_router"], dtype=np.float64)
    d_router = np.zeros_like(W_r)
    for t in range(T):
        for k in range(K):
            e = int(ids[t, k])
            d_router[e] += dz[t, k] * x[t]
            dx[t] += dz[t, k] * W_r[e]
    if "w_sh_up" in weights:
        W_su = np.asarray(weights["w_sh_up"], dtype=np.float64)
        W_sd = np.asarray(weights["w_sh_down"], dtype=np.float64)
        a_s = rnd(x @ W_su.T)
        h_s = rnd(np.maximum(a_s, 0.0) ** 2)
        out["d_w_sh_down"] = D.T @ h_s
        if bf16_points:
            da_s = rnd((D @ W_sd) * 2.0 * np.sqrt(h_s))
        else:
            da_s = (D @ W_sd) * 2.0 * np.maximum(a_s, 0.0)
        out["d_w_sh_up"] = da_s.T @ x
        dx += da_s @ W_su
    if latent:
        dx_l = rnd(dx_e)
        out["d_w_lat_down"] = dx_l.T @ x
        dx += dx_l @ W_ld
    else:
        dx += dx_e
    out.update({"dx": dx, "d_w_router": d_router, "d_w_up": d_up, "d_w_down": d_down, "q": q, "ds": ds,
                "dz": dz, "w": w, "y_routed": y_r})
    return out


def rms_norm_backward(x: np.ndarray, gamma: np.ndarray, eps: float, dxn: np.ndarray):
    """(dx, dgamma) of xn = gamma * x r, r = 1 / sqrt(mean(x^2) + eps):
    dx_i = r gamma_i dxn_i - r^3 x_i / d * sum_j gamma_j dxn_j x_j;
    dgamma = sum over rows of dxn * x r."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64)[None, :]
    dxn = np.asarray(dxn, dtype=np.float64)
    d = x.shape[1]
    r = 1.0 / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)
    dot = np.sum(g * dxn * x, axis=1, keepdims=True)
    dx = r * g * dxn - r ** 3 * x * dot / d
    return dx, np.sum(dxn * x * r, axis=0)


def block_backward(x: np.ndarray, gamma: np.ndarray, eps: float, weights: Dict[str, np.ndarray],
                   ids: np.ndarray, scores: np.ndarray, dout: np.ndarray, n_experts: int,
                   norm_topk_prob: int, rsf: float, xn: Optional[np.ndarray] = None,
                   bf16_points: bool = False) -> Dict[str, object]:
    """Gradients of L = <dout, out> for out = x + layer(RMSNorm(x)) with the
    routing frozen: the residual passes dout to x unchanged (page section
    0x06F.6: the residual is the third path into the block input), the layer's
    input gradient goes back through the RMSNorm.  ``xn``: the normalised rows
    the layer read (as the device stored them), else the float64 RMSNorm."""
    xn_v = rms_norm(x, gamma, eps) if xn is None else np.asarray(xn, dtype=np.float64)
    out = layer_backward(xn_v, weights, ids, scores, dout, n_experts, norm_topk_prob, rsf, bf16_points)
    dxn = out["dx"]
    dx, dgamma = rms_norm_backward(x, gamma, eps, dxn)
    out["dxn"] = dxn
    out["dx"] = np.asarray(dout, dtype=np.float64) + dx
    out["d_norm_w"] = dgamma
    return out


class _LazyExpert:
    """Expert e as a callable (matrices fetched, and dequantised, on first use)."""

    def __init__(self, weights, e, bf16_points, act_terms=None):
        self.weights, self.e, self.bf16_points, self.act_terms = weights, e, bf16_points, act_terms

    def __call__(self, xs: np.ndarray) -> np.ndarray:
        up, down = expert_matrices(self.weights, self.e)
        return relu2_mlp(xs, up, down, self.bf16_points, self.act_terms)


def full_layer(x: np.ndarray, weights: Dict[str, np.ndarray], n_experts: int, top_k: int,
               n_group: int, topk_group: int, norm_topk_prob: int, rsf: float,
               bf16_points: bool, logits_f32: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Whole layer from hidden rows: router (on ``logits_f32`` if given, else on the
    oracle's own logits rounded to FP32), selection, weights, experts, combine."""
    z, zscale = router_logits(x, weights["w_router"])
    zl = np.asarray(logits_f32, dtype=np.float32) if logits_f32 is not None else z.astype(np.float32)
    s = sigmoid_scores(zl)
    ids, w = route(s, weights.get("bias"), n_group, topk_group, top_k, norm_topk_prob, rsf)
    out = layer_forward(x, weights, ids, w, n_experts, bf16_points)
    out.update({"logits": z, "logit_scale": zscale, "scores": s, "ids": ids, "w": w})
    return out
