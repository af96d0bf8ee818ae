// Router selection for one token by one warp (page "Nemotron Is Not One
// Circuit: Mamba, Attention, and MoE Routing", sections "The Router Is A
// Deterministic Algorithm" and "The C Kernel Contract"; page "NemotronH
// (Nemotron 3.5 Lightning, Bolt, Super VL)", section "Arithmetic").  Shared by
// the selection kernel and the fused selection + dispatch kernel for a few
// tokens.
#pragma once

#include "internal.h"

#include <climits>

namespace moe {

// ---------------------------------------------------------------------------
// selection: one warp per token; lane l holds the P consecutive experts
// lP .. lP+P-1, so experts ascend with the lane and, where P divides the group
// size, a group is a run of lanes.
// Ordering key: larger biased score first, NaN after every number, equal keys
// to the lower expert id.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int order_key(float v) {
  if (isnan(v)) return INT_MIN + 1;
  v = v + 0.0f;  // -0 -> +0
  const int b = __float_as_int(v);
  return b >= 0 ? b : (b ^ 0x7FFFFFFF);
}

__device__ __forceinline__ bool better(int ka, int ea, int kb, int eb) {
  return ka > kb || (ka == kb && ea < eb);
}

// top two (key, id, value) of a lane's candidates, then merged across the
// lanes whose xor distance is below `span` (a power of two)
struct Top2 {
  int k1, e1, k2, e2;
  float v1, v2;
};
__device__ __forceinline__ void top2_add(Top2& t, int k, int e, float v) {
  if (better(k, e, t.k1, t.e1)) {
    t.k2 = t.k1; t.e2 = t.e1; t.v2 = t.v1;
    t.k1 = k; t.e1 = e; t.v1 = v;
  } else if (better(k, e, t.k2, t.e2)) {
    t.k2 = k; t.e2 = e; t.v2 = v;
  }
}
__device__ __forceinline__ void top2_merge(Top2& t, int span) {
  for (int off = span >> 1; off > 0; off >>= 1) {
    Top2 o;
    o.k1 = __shfl_xor_sync(0xffffffffu, t.k1, off); o.e1 = __shfl_xor_sync(0xffffffffu, t.e1, off);
    o.k2 = __shfl_xor_sync(0xffffffffu, t.k2, off); o.e2 = __shfl_xor_sync(0xffffffffu, t.e2, off);
    o.v1 = __shfl_xor_sync(0xffffffffu, t.v1, off); o.v2 = __shfl_xor_sync(0xffffffffu, t.v2, off);
    // both inputs are ordered pairs: the result is the best two of the four
    if (better(o.k1, o.e1, t.k1, t.e1)) {
      if (better(t.k1, t.e1, o.k2, o.e2)) { t.k2 = t.k1; t.e2 = t.e1; t.v2 = t.v1; }
      else { t.k2 = o.k2; t.e2 = o.e2; t.v2 = o.v2; }
      t.k1 = o.k1; t.e1 = o.e1; t.v1 = o.v1;
    } else if (better(o.k1, o.e1, t.k2, t.e2)) {
      t.k2 = o.k1; t.e2 = o.e1; t.v2 = o.v1;
    }
  }
}

// Top-K of a warp's candidates for K > 8 (K <= 32), by selection instead of K
// rounds of maxima: the ordering keys, as unsigned numbers (non-candidates 0,
// every candidate at least 1), give the K-th largest key thr by a bitwise
// search from the highest bit where the candidates differ (a warp-wide count of
// keys >= a trial value per bit); the chosen are the keys above thr and, of
// the keys equal to it, the lowest ids (values ascend in id across lanes and
// within a lane); a chosen value's slot is the number of chosen values ahead of
// it in (key descending, id ascending) order.  Same ids, slots and weights as
// the rounds (the weight sum still runs in slot order).
template <int P>
__device__ __forceinline__ void topk_radix(const int (&key)[P], uint32_t cand, const float (&s)[P], int e0, int E,
                                           int K, int norm, float rsf, int t, int32_t* __restrict__ ids,
                                           float* __restrict__ wout, int warp, int lane) {
  __shared__ uint32_t sel_key[32][32];
  __shared__ int sel_e[32][32];
  __shared__ float sel_s[32][32];
  __shared__ float slot_s[32][32];
  constexpr unsigned FULL = 0xffffffffu;
  uint32_t uk[P];
  uint32_t lmax = 0u, lmin = 0xffffffffu;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const bool ok = ((cand >> j) & 1u) && e0 + j < E;
    uk[j] = ok ? ((uint32_t)key[j] ^ 0x80000000u) : 0u;
    if (ok) {
      lmax = max(lmax, uk[j]);
      lmin = min(lmin, uk[j]);
    }
  }
  const uint32_t hi = __reduce_max_sync(FULL, lmax), lo = __reduce_min_sync(FULL, lmin);
  // the K-th largest key lies in [lo, hi]: it shares their common high bits
  const int top = hi == lo ? -1 : 31 - __clz(hi ^ lo);
  uint32_t thr = top < 0 ? hi : (top == 31 ? 0u : (hi & ~((2u << top) - 1u)));
  for (int b = top; b >= 0; --b) {
    const uint32_t trial = thr | (1u << b);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < P; ++j) cnt += uk[j] >= trial ? 1 : 0;
    if (__reduce_add_sync(FULL, cnt) >= K) thr = trial;
  }
  int ngt = 0, neq = 0;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    ngt += uk[j] > thr ? 1 : 0;
    neq += uk[j] == thr ? 1 : 0;
  }
  const int need = K - __reduce_add_sync(FULL, ngt);      // >= 1 keys equal to thr are taken
  int pre = neq;                                          // equal keys in lower lanes
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(FULL, pre, off);
    if (lane >= off) pre += v;
  }
  pre -= neq;
  uint32_t take = 0u;
  int nsel = 0;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const bool eq = uk[j] == thr;
    if (uk[j] > thr || (eq && pre < need)) {
      take |= 1u << j;
      ++nsel;
    }
    if (eq) ++pre;
  }
  int base = nsel;                                        // chosen values in lower lanes
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(FULL, base, off);
    if (lane >= off) base += v;
  }
  base -= nsel;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    if ((take >> j) & 1u) {
      sel_key[warp][base] = uk[j];
      sel_e[warp][base] = e0 + j;
      sel_s[warp][base] = s[j];
      ++base;
    }
  }
  __syncwarp();
  int rank = 0, ei = 0;
  float si = 0.f;
  if (lane < K) {
    const uint32_t ki = sel_key[warp][lane];
    ei = sel_e[warp][lane];
    si = sel_s[warp][lane];
    for (int j = 0; j < K; ++j) {
      const uint32_t kj = sel_key[warp][j];
      rank += (kj > ki || (kj == ki && sel_e[warp][j] < ei)) ? 1 : 0;
    }
    slot_s[warp][rank] = si;
  }
  __syncwarp();
  float wsum = 0.f;
  for (int k = 0; k < K; ++k) wsum += slot_s[warp][k];   // slot order, FP32
  if (lane < K) {
    const float wv = norm ? (si / wsum) * rsf : si * rsf;
    ids[(int64_t)t * K + rank] = ei;
    wout[(int64_t)t * K + rank] = wv;
  }
  __syncwarp();          // the shared rows are reused by this warp's next token
}

// One token's selection, by one warp (lane = its lane, warp = its warp index in
// the CTA).  logits: slab 0 of nparts slabs part_stride floats apart.
template <int P>
__device__ __forceinline__ void select_token(const float* __restrict__ logits, int nparts, int64_t part_stride,
                                             float* __restrict__ logits_out, int t, int E,
                                             const float* __restrict__ bias, int G, int TG, int K, int norm,
                                             float rsf, float* __restrict__ scores, int32_t* __restrict__ ids,
                                             float* __restrict__ wout, int32_t* err, int warp, int lane,
                                             bool radix) {
  const int e0 = lane * P;
  float s[P], c[P];
  int key[P];
  bool any_nan = false;
  const float* zrow = logits + (int64_t)t * E;
  float* srow = scores + (int64_t)t * E;
  // every load first (logits, their K parts, the bias), then the arithmetic,
  // then the stores: interleaved, each store would order the next load behind it
  float zv[P], bv[P];
  if (P % 4 == 0 && E == 32 * P) {
    // every lane full: 16-byte loads (rows of E floats, E a multiple of 4)
#pragma unroll
    for (int j = 0; j < P; j += 4) {
      const float4 z4 = *reinterpret_cast<const float4*>(zrow + e0 + j);
      zv[j] = z4.x; zv[j + 1] = z4.y; zv[j + 2] = z4.z; zv[j + 3] = z4.w;
      const float4 b4 = bias ? *reinterpret_cast<const float4*>(bias + e0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      bv[j] = b4.x; bv[j + 1] = b4.y; bv[j + 2] = b4.z; bv[j + 3] = b4.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const int e = e0 + j;
      zv[j] = e < E ? zrow[e] : 0.f;
      bv[j] = (bias && e < E) ? bias[e] : 0.f;
    }
  }
  for (int p = 1; p < nparts; ++p) {
#pragma unroll
    for (int j = 0; j < P; ++j)
      if (e0 + j < E) zv[j] += zrow[p * part_stride + e0 + j];   // K parts added in part order
  }
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const int e = e0 + j;
    if (e < E) {
      const float sv = 1.0f / (1.0f + expf(-zv[j]));
      s[j] = sv;
      const float cv = bias ? sv + bv[j] : sv;
      c[j] = cv;
      key[j] = order_key(cv);
      any_nan |= isnan(cv);
    } else {
      s[j] = 0.f;
      c[j] = 0.f;
      key[j] = INT_MIN;  // not an expert: never chosen
    }
  }
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const int e = e0 + j;
    if (e < E) {
      srow[e] = s[j];
      if (logits_out) logits_out[(int64_t)t * E + e] = zv[j];
    }
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) set_error(err, MOE_DEVERR_NONFINITE);

  // group limit: keep the TG groups with the largest sum of their two largest
  // c (ties to the lower group); cand bit j = value j may be chosen
  uint32_t cand = 0xffffffffu;
  if (G > 1 && TG < G) {
    const int gsz = E / G;
    const int lpg = gsz / P;                       // lanes per group when P divides gsz
    if (gsz % P == 0 && (lpg & (lpg - 1)) == 0) {
      // each lane lies in one group g = lane / lpg: lane top two, merged over the group's lanes
      const int g = lane / lpg;
      Top2 tp{INT_MIN, INT_MAX, INT_MIN, INT_MAX, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < P; ++j)
        if (e0 + j < E) top2_add(tp, key[j], e0 + j, c[j]);
      top2_merge(tp, lpg);
      const float gs = tp.v1 + tp.v2;
      const int gk = order_key(gs);
      // rank of this lane's group among all G group scores
      int rank = 0;
      for (int g2 = 0; g2 < G; ++g2) {
        const int k2 = __shfl_sync(0xffffffffu, gk, g2 * lpg);
        rank += better(k2, g2, gk, g) ? 1 : 0;
      }
      cand = (g < G && rank < TG) ? 0xffffffffu : 0u;
    } else {
      // general layout: one pass per group over every lane's values
      __shared__ float gsum_sh[32][32];
      float* gsum = gsum_sh[warp];
      uint32_t kept = 0;
#pragma unroll 1
      for (int g = 0; g < G; ++g) {
        Top2 tp{INT_MIN, INT_MAX, INT_MIN, INT_MAX, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const int e = e0 + j;
          if (e < E && e / gsz == g) top2_add(tp, key[j], e, c[j]);
        }
        top2_merge(tp, 32);
        if (lane == 0) gsum[g] = tp.v1 + tp.v2;
      }
      __syncwarp();
#pragma unroll 1
      for (int n = 0; n < TG; ++n) {
        int bk = INT_MIN, bg = INT_MAX;
#pragma unroll 1
        for (int g = 0; g < G; ++g) {
          if (!((kept >> g) & 1u)) {
            const int kg = order_key(gsum[g]);
            if (better(kg, g, bk, bg)) { bk = kg; bg = g; }
          }
        }
        kept |= 1u << bg;
      }
      cand = 0;
#pragma unroll
      for (int j = 0; j < P; ++j)
        if (e0 + j < E && ((kept >> ((e0 + j) / gsz)) & 1u)) cand |= 1u << j;
    }
  }

  // above 8 chosen experts and 8 tokens the threshold search beat the rounds
  // (16 tokens of a 22-of-512 router: 7 us less a layer); at 8 tokens and
  // fewer the rounds measured 1-4 us faster
  if (radix && K > 8) {
    topk_radix<P>(key, cand, s, e0, E, K, norm, rsf, t, ids, wout, warp, lane);
    return;
  }

  // top-K: every lane keeps the best of its remaining candidates; each round
  // the warp maximum of the lane keys (ties: the lowest lane, which holds the
  // lowest ids) wins and only the winning lane looks again among its values
  uint32_t taken = 0;
  float wsel = 0.f;          // lane k keeps the score of slot k
  int esel = 0;
  float wsum = 0.f;
  int lk = INT_MIN, lj = -1;
  auto rescan = [&]() {
    lk = INT_MIN; lj = -1;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      if (((cand & ~taken) >> j) & 1u && key[j] > lk && e0 + j < E) { lk = key[j]; lj = j; }
    }
  };
  rescan();
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    const int mk = __reduce_max_sync(0xffffffffu, lk);
    const uint32_t hit = __ballot_sync(0xffffffffu, lk == mk && lj >= 0);
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j)
      if (j == lj) ls = s[j];
    int be = INT_MAX;
    float bs = 0.f;
    if (hit) {
      const int src = __ffs(hit) - 1;
      be = __shfl_sync(0xffffffffu, e0 + lj, src);
      bs = __shfl_sync(0xffffffffu, ls, src);
      if (lane == src) {
        taken |= 1u << lj;
        rescan();
      }
    }
    if (lane == k) { wsel = bs; esel = be; }
    wsum += bs;              // slot order, FP32
  }
  if (lane < K) {
    const float wv = norm ? (wsel / wsum) * rsf : wsel * rsf;
    ids[(int64_t)t * K + lane] = esel;
    wout[(int64_t)t * K + lane] = wv;
  }
}



// ---------------------------------------------------------------------------
// One token's selection by a whole CTA of NT threads (E <= NT, K <= 32; with a
// group limit, groups of a multiple of 32 experts, at most 32 groups): thread
// i holds expert i, so the loads, sigmoids and stores take one step instead
// of P per lane.  Every value that decides or is stored comes from the same
// expressions in the same order as select_token: the group score is the sum
// of the group's two best biased scores, the K-th largest ordering key is
// found bit by bit (a CTA-wide count per bit), keys above it are chosen and,
// of the keys equal to it, the lowest ids; slots are (key descending, id
// ascending) and the weight sum runs in slot order.  Every thread of the CTA
// calls it (it holds CTA barriers).
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ bool cta_select_fits(int NT, int E, int G, int TG, int K) {
  return E <= NT && K <= 32 && (G <= 1 || TG >= G || (G <= 32 && E % G == 0 && (E / G) % 32 == 0));
}

template <int NT>
__device__ __forceinline__ void select_token_cta(const float* __restrict__ logits, int nparts, int64_t part_stride,
                                                 float* __restrict__ logits_out, int t, int E,
                                                 const float* __restrict__ bias, int G, int TG, int K, int norm,
                                                 float rsf, float* __restrict__ scores, int32_t* __restrict__ ids,
                                                 float* __restrict__ wout, int32_t* err) {
  constexpr int NW = NT / 32;
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ int c_k1[NW], c_e1[NW], c_k2[NW], c_e2[NW];
  __shared__ float c_v1[NW], c_v2[NW];
  __shared__ int c_gkey[32];
  __shared__ int c_cnt[NW];
  __shared__ uint32_t c_sel_key[32];
  __shared__ int c_sel_e[32];
  __shared__ float c_sel_s[32], c_slot_s[32];
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const bool live = i < E;
  float sv = 0.f, cv = 0.f;
  int key = INT_MIN;
  if (live) {
    const float* zrow = logits + (int64_t)t * E;
    float z = zrow[i];
    for (int p = 1; p < nparts; ++p) z += zrow[p * part_stride + i];   // K parts added in part order
    sv = 1.0f / (1.0f + expf(-z));
    cv = bias ? sv + bias[i] : sv;
    key = order_key(cv);
    scores[(int64_t)t * E + i] = sv;
    if (logits_out) logits_out[(int64_t)t * E + i] = z;
  }
  if (__syncthreads_or(live && isnan(cv)) && i == 0) set_error(err, MOE_DEVERR_NONFINITE);

  // group limit: each warp's best two, merged per group, ranked
  bool cand = live;
  if (G > 1 && TG < G) {
    const int gsz = E / G, wpg = gsz / 32;
    Top2 tp{INT_MIN, INT_MAX, INT_MIN, INT_MAX, 0.f, 0.f};
    if (live) top2_add(tp, key, i, cv);
    top2_merge(tp, 32);
    if (lane == 0) {
      c_k1[warp] = tp.k1; c_e1[warp] = tp.e1; c_v1[warp] = tp.v1;
      c_k2[warp] = tp.k2; c_e2[warp] = tp.e2; c_v2[warp] = tp.v2;
    }
    __syncthreads();
    if (i < G) {
      Top2 g2{INT_MIN, INT_MAX, INT_MIN, INT_MAX, 0.f, 0.f};
      for (int w = i * wpg; w < (i + 1) * wpg; ++w) {
        top2_add(g2, c_k1[w], c_e1[w], c_v1[w]);
        top2_add(g2, c_k2[w], c_e2[w], c_v2[w]);
      }
      c_gkey[i] = order_key(g2.v1 + g2.v2);
    }
    __syncthreads();
    if (live) {
      const int g = i / gsz, gk = c_gkey[g];
      int rank = 0;
      for (int g2 = 0; g2 < G; ++g2) rank += better(c_gkey[g2], g2, gk, g) ? 1 : 0;
      cand = rank < TG;
    }
  }

  // the K-th largest key among the candidates (as unsigned numbers, every
  // candidate at least 1): the largest value with at least K keys at or above it
  const uint32_t uk = cand ? ((uint32_t)key ^ 0x80000000u) : 0u;
  uint32_t thr = 0u;
  for (int b = 31; b >= 0; --b) {
    const uint32_t trial = thr | (1u << b);
    if (__syncthreads_count(cand && uk >= trial) >= K) thr = trial;
  }
  const int need = K - __syncthreads_count(cand && uk > thr);   // >= 1 keys equal to thr are taken
  const bool eq = cand && uk == thr;
  const uint32_t eqm = __ballot_sync(FULL, eq);
  if (lane == 0) c_cnt[warp] = __popc(eqm);
  __syncthreads();
  int pre = __popc(eqm & ((1u << lane) - 1u));                   // equal keys at lower ids
  for (int w = 0; w < warp; ++w) pre += c_cnt[w];
  const bool take = cand && (uk > thr || (eq && pre < need));
  const uint32_t tm = __ballot_sync(FULL, take);
  __syncthreads();                                              // every thread has read c_cnt
  if (lane == 0) c_cnt[warp] = __popc(tm);
  __syncthreads();
  if (take) {
    int pos = __popc(tm & ((1u << lane) - 1u));                 // K chosen in id order
    for (int w = 0; w < warp; ++w) pos += c_cnt[w];
    c_sel_key[pos] = uk;
    c_sel_e[pos] = i;
    c_sel_s[pos] = sv;
  }
  __syncthreads();
  if (warp == 0) {
    int rank = 0, ei = 0;
    float si = 0.f;
    if (lane < K) {
      const uint32_t ki = c_sel_key[lane];
      ei = c_sel_e[lane];
      si = c_sel_s[lane];
      for (int j = 0; j < K; ++j) {
        const uint32_t kj = c_sel_key[j];
        rank += (kj > ki || (kj == ki && c_sel_e[j] < ei)) ? 1 : 0;
      }
      c_slot_s[rank] = si;
    }
    __syncwarp();
    float wsum = 0.f;
    for (int k = 0; k < K; ++k) wsum += c_slot_s[k];            // slot order, FP32
    if (lane < K) {
      const float wv = norm ? (si / wsum) * rsf : si * rsf;
      ids[(int64_t)t * K + rank] = ei;
      wout[(int64_t)t * K + rank] = wv;
    }
  }
}

}  // namespace moe
