// Router: FP32 logits, FP32 sigmoid scores, group-limited top-k selection,
// routing weights (page "Nemotron Is Not One Circuit: Mamba, Attention, and
// MoE Routing", sections "The Router Is A Deterministic Algorithm" and "The C
// Kernel Contract"; page "NemotronH (Nemotron 3.5 Lightning, Bolt, Super VL)",
// section "Arithmetic": fp32 logits, sigmoid, the bias for the choice only,
// ties to the lower id).
#include "internal.h"

#include <algorithm>
#include <climits>

namespace moe {

namespace {

// ---------------------------------------------------------------------------
// logits, few tokens: a CTA computes EPC experts x TMAX tokens; its 8 warps are
// EPC experts x (8 / EPC) interleaved K slices of 256, each lane an FP32 FMA
// chain over 8 consecutive elements; lanes reduce by a fixed shuffle tree and
// the K slices by a fixed order through shared memory.  W_r rows are streamed
// once per token group; the token rows are shared by the CTA's experts in L1.
// ---------------------------------------------------------------------------
template <int TMAX, int EPC, bool XF32>
__global__ void __launch_bounds__(256) router_logits_small(const void* __restrict__ X, int T, int d,
                                                           const float* __restrict__ Wr, int E,
                                                           float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  constexpr int KS = 8 / EPC;
  __shared__ float red[8][TMAX];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ei = warp % EPC, ks = warp / EPC;
  const int e = blockIdx.x * EPC + ei;
  const int t0 = blockIdx.y * TMAX;
  const int nt = min(TMAX, T - t0);
  float acc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
  if (e < E) {
    const float* w = Wr + (int64_t)e * d;
#pragma unroll 2
    for (int k = ks * 256 + lane * 8; k < d; k += KS * 256) {
      const uint4 wa = ldg_stream(w + k);
      const uint4 wb = ldg_stream(w + k + 4);
      const float wv[8] = {__uint_as_float(wa.x), __uint_as_float(wa.y), __uint_as_float(wa.z),
                           __uint_as_float(wa.w), __uint_as_float(wb.x), __uint_as_float(wb.y),
                           __uint_as_float(wb.z), __uint_as_float(wb.w)};
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < nt) {
          float xv[8];
          if (XF32) {
            const float* xp = reinterpret_cast<const float*>(X) + (int64_t)(t0 + t) * d + k;
            const float4 a = *reinterpret_cast<const float4*>(xp);
            const float4 b = *reinterpret_cast<const float4*>(xp + 4);
            xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
            xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
          } else {
            const uint4 q = ldg_keep(reinterpret_cast<const bf16*>(X) + (int64_t)(t0 + t) * d + k);
            xv[0] = bf16_lo(q.x); xv[1] = bf16_hi(q.x); xv[2] = bf16_lo(q.y); xv[3] = bf16_hi(q.y);
            xv[4] = bf16_lo(q.z); xv[5] = bf16_hi(q.z); xv[6] = bf16_lo(q.w); xv[7] = bf16_hi(q.w);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[t] = fmaf(xv[i], wv[i], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    float v = acc[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) red[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < EPC * TMAX) {
    const int eo = threadIdx.x / TMAX, t = threadIdx.x % TMAX;
    const int ee = blockIdx.x * EPC + eo;
    if (ee < E && t < nt) {
      float v = 0.f;
      for (int k2 = 0; k2 < KS; ++k2) v += red[k2 * EPC + eo][t];
      logits[(int64_t)(t0 + t) * E + ee] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// logits, many tokens: shared-memory tiled FP32 GEMM, 64 tokens x 64 experts
// per CTA, 4x4 outputs per thread, K slices of 16.
// ---------------------------------------------------------------------------
template <bool XF32>
__global__ void __launch_bounds__(256) router_logits_tiled(const void* __restrict__ X, int T, int d,
                                                           const float* __restrict__ Wr, int E,
                                                           float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  __shared__ float xs[16][64 + 4];
  __shared__ float ws[16][64 + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int ty = tid >> 4, tx = tid & 15;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += 16) {
    // each thread loads 4 x and 4 w values: row = tid / 4, k sub = (tid % 4) * 4
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    {
      const int t = t0 + lr;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < T) {
        if (XF32) {
          const float4 q = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(X) + (int64_t)t * d + k0 + lk);
          v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else {
          const uint2 q = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(X) + (int64_t)t * d + k0 + lk);
          v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) xs[lk + i][lr] = v[i];
      const int e = e0 + lr;
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) q = *reinterpret_cast<const float4*>(Wr + (int64_t)e * d + k0 + lk);
      ws[lk + 0][lr] = q.x; ws[lk + 1][lr] = q.y; ws[lk + 2][lr] = q.z; ws[lk + 3][lr] = q.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float xa[4], wb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { xa[i] = xs[kk][ty * 4 + i]; wb[i] = ws[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[(int64_t)t * E + e] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// selection: one warp per token, lane l holds experts l, l+32, ...
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

template <int P>
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ logits, int T, int E,
                                                            const float* __restrict__ bias, int G, int TG,
                                                            int K, int norm, float rsf,
                                                            float* __restrict__ scores,
                                                            int32_t* __restrict__ ids,
                                                            float* __restrict__ wout,
                                                            int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float s[P], c[P];
  int key[P];
  bool any_nan = false;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const int e = lane + 32 * j;
    if (e < E) {
      const float z = logits[(int64_t)t * E + e];
      const float sv = 1.0f / (1.0f + expf(-z));
      s[j] = sv;
      scores[(int64_t)t * E + e] = sv;
      const float cv = bias ? sv + bias[e] : sv;
      c[j] = cv;
      key[j] = order_key(cv);
      any_nan |= isnan(cv);
    } else {
      s[j] = 0.f;
      c[j] = 0.f;
      key[j] = INT_MIN;  // not an expert: never chosen
    }
  }
  if (__any_sync(0xffffffffu, any_nan) && lane == 0) set_error(err, MOE_DEVERR_NONFINITE);

  // group of each held expert (one division per held value)
  const int gsz = E / G;
  int grp[P];
#pragma unroll
  for (int j = 0; j < P; ++j) grp[j] = (lane + 32 * j) / gsz;

  // group limit: keep the TG groups with the largest sum of their two largest c
  uint32_t kept = 0xffffffffu;
  if (G > 1 && TG < G) {
    float gsum[32];
#pragma unroll
    for (int g = 0; g < 32; ++g) gsum[g] = 0.f;
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
      int k1 = INT_MIN, e1 = INT_MAX, k2 = INT_MIN, e2 = INT_MAX;
      float v1 = 0.f, v2 = 0.f;
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const int e = lane + 32 * j;
        if (e < E && grp[j] == g) {
          if (better(key[j], e, k1, e1)) {
            k2 = k1; e2 = e1; v2 = v1;
            k1 = key[j]; e1 = e; v1 = c[j];
          } else if (better(key[j], e, k2, e2)) {
            k2 = key[j]; e2 = e; v2 = c[j];
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const int ok1 = __shfl_xor_sync(0xffffffffu, k1, off), oe1 = __shfl_xor_sync(0xffffffffu, e1, off);
        const int ok2 = __shfl_xor_sync(0xffffffffu, k2, off), oe2 = __shfl_xor_sync(0xffffffffu, e2, off);
        const float ov1 = __shfl_xor_sync(0xffffffffu, v1, off), ov2 = __shfl_xor_sync(0xffffffffu, v2, off);
        // merge two sorted pairs into the top two
        if (better(ok1, oe1, k1, e1)) {
          if (better(k1, e1, ok2, oe2)) { k2 = k1; e2 = e1; v2 = v1; }
          else { k2 = ok2; e2 = oe2; v2 = ov2; }
          k1 = ok1; e1 = oe1; v1 = ov1;
        } else if (better(ok1, oe1, k2, e2)) {
          k2 = ok1; e2 = oe1; v2 = ov1;
        }
      }
      // (g is warp-uniform: the select below keeps gsum in registers)
#pragma unroll
      for (int gg = 0; gg < 32; ++gg)
        if (gg == g) gsum[gg] = v1 + v2;
    }
    kept = 0;
#pragma unroll 1
    for (int n = 0; n < TG; ++n) {
      int bk = INT_MIN, bg = INT_MAX;
#pragma unroll
      for (int g = 0; g < 32; ++g) {
        if (g < G && !((kept >> g) & 1u)) {
          const int kg = order_key(gsum[g]);
          if (better(kg, g, bk, bg)) { bk = kg; bg = g; }
        }
      }
      kept |= 1u << bg;
    }
  }

  // top-K among experts of kept groups: every lane keeps the best of its own
  // remaining candidates; each round the warp takes the best lane-best and only
  // the winning lane looks again among its values
  uint32_t taken = 0;
  float wsel = 0.f;          // lane k keeps the score of slot k
  int esel = 0;
  float wsum = 0.f;
  int lk = INT_MIN, le = INT_MAX;
  float ls = 0.f;
  auto rescan = [&]() {
    lk = INT_MIN; le = INT_MAX; ls = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && ((kept >> grp[j]) & 1u)) {
        if (better(key[j], e, lk, le)) { lk = key[j]; le = e; ls = s[j]; }
      }
    }
  };
  rescan();
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    int bk = lk, be = le;
    float bs = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const int ok = __shfl_xor_sync(0xffffffffu, bk, off), oe = __shfl_xor_sync(0xffffffffu, be, off);
      const float os = __shfl_xor_sync(0xffffffffu, bs, off);
      if (better(ok, oe, bk, be)) { bk = ok; be = oe; bs = os; }
    }
    if (lane == k) { wsel = bs; esel = be; }
    wsum += bs;              // slot order, FP32
    if (be != INT_MAX && (be & 31) == lane) {
      taken |= 1u << (be >> 5);
      rescan();
    }
  }
  if (lane < K) {
    const float wv = norm ? (wsel / wsum) * rsf : wsel * rsf;
    ids[(int64_t)t * K + lane] = esel;
    wout[(int64_t)t * K + lane] = wv;
  }
}

// W (FP32) -> [W1 | W2 | W3] (BF16, side by side along K): W1 = bf16(W),
// W2 = bf16(W - W1), W3 = bf16(W - W1 - W2).  Each difference is exact in FP32
// and each term keeps 8 more significand bits, so sum(x * Wi) with FP32
// accumulation carries FP32-level precision for BF16 x (exact in BF16).
__global__ void split_bf16x3_kernel(const float* __restrict__ w, int E, int d, bf16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = (int64_t)E * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / d, j = i - e * d;
    const float v = w[i];
    const bf16 w1 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(w1);
    const bf16 w2 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(w2);
    const bf16 w3 = __float2bfloat16_rn(r2);
    bf16* row = out + e * 3 * (int64_t)d;
    row[j] = w1;
    row[d + j] = w2;
    row[2 * (int64_t)d + j] = w3;
  }
}

template <int P>
cudaError_t launch_select_p(const float* logits, int T, int E, const float* bias, int G, int TG, int K,
                            int norm, float rsf, float* scores, int32_t* ids, float* w, int32_t* err,
                            cudaStream_t s) {
  launch_k(router_select_kernel<P>, (unsigned)ceil_div(T, 8), 256, 0, s, logits, T, E, bias, G, TG, K, norm, rsf,
                                                                   scores, ids, w, err);
  return cudaGetLastError();
}

template <int TMAX, int EPC>
cudaError_t launch_small_t(const void* x, int act, int T, int d, const float* w, int E, float* logits,
                           cudaStream_t s) {
  dim3 grid((unsigned)ceil_div(E, EPC), (unsigned)ceil_div(T, TMAX));
  if (act == MOE_DT_F32)
    launch_k(router_logits_small<TMAX, EPC, true>, grid, 256, 0, s, x, T, d, w, E, logits);
  else
    launch_k(router_logits_small<TMAX, EPC, false>, grid, 256, 0, s, x, T, d, w, E, logits);
  return cudaGetLastError();
}

template <int TMAX>
cudaError_t launch_small(const void* x, int act, int T, int d, const float* w, int E, float* logits,
                         cudaStream_t s) {
  // wide routers share each CTA's token rows among several experts
  if (E >= 256) return launch_small_t<TMAX, 2>(x, act, T, d, w, E, logits, s);
  return launch_small_t<TMAX, 1>(x, act, T, d, w, E, logits, s);
}

}  // namespace

cudaError_t launch_router_logits(const void* x, int act, int T, int d, const float* w_router, int E,
                                 float* logits, cudaStream_t s, void* w_split) {
  if (T <= 0) return cudaSuccess;
  if (w_split && act == MOE_DT_BF16 && T > 64 && E % 32 == 0 && d % 64 == 0) {
    const int64_t n = (int64_t)E * d;
    launch_k(split_bf16x3_kernel, (unsigned)std::min<int64_t>(ceil_div(n, 256), 2048), 256, 0, s, w_router, E, d, reinterpret_cast<bf16*>(w_split));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    GemvArgs a{};
    a.W = w_split; a.N = E; a.K = 3 * d; a.X = x; a.x_ld = d; a.dense_rows = T;
    a.out = logits; a.out_ld = E;
    const int bn = T >= 64 * 152 ? 64 : 32;
    return launch_gemm_tc(a, EPI_STORE, true, E, T, 0, bn, s, d);
  }
  if (T <= 4) return launch_small<4>(x, act, T, d, w_router, E, logits, s);
  if (T <= 64) return launch_small<8>(x, act, T, d, w_router, E, logits, s);
  dim3 grid((unsigned)ceil_div(T, 64), (unsigned)ceil_div(E, 64));
  if (act == MOE_DT_F32)
    launch_k(router_logits_tiled<true>, grid, 256, 0, s, x, T, d, w_router, E, logits);
  else
    launch_k(router_logits_tiled<false>, grid, 256, 0, s, x, T, d, w_router, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_router_select(const float* logits, int T, int E, const float* bias, int G, int TG, int K,
                                 int norm, float rsf, float* scores, int32_t* ids, float* w, int32_t* err,
                                 cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int P = (int)ceil_div(E, 32);
  if (P <= 1) return launch_select_p<1>(logits, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, err, s);
  if (P <= 2) return launch_select_p<2>(logits, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, err, s);
  if (P <= 4) return launch_select_p<4>(logits, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, err, s);
  if (P <= 8) return launch_select_p<8>(logits, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, err, s);
  if (P <= 16) return launch_select_p<16>(logits, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, err, s);
  return launch_select_p<32>(logits, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, err, s);
}

}  // namespace moe
