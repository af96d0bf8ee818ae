// Router: FP32 logits, FP32 sigmoid scores, group-limited top-k selection,
// routing weights (page "Nemotron Is Not One Circuit: Mamba, Attention, and
// MoE Routing", sections "The Router Is A Deterministic Algorithm" and "The C
// Kernel Contract"; page "NemotronH (Nemotron 3.5 Lightning, Bolt, Super VL)",
// section "Arithmetic": fp32 logits, sigmoid, the bias for the choice only,
// ties to the lower id).
#include "select.cuh"

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

template <int P>
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ logits, int nparts,
                                                            int64_t part_stride, float* __restrict__ logits_out,
                                                            int T, int E,
                                                            const float* __restrict__ bias, int G, int TG,
                                                            int K, int norm, float rsf,
                                                            float* __restrict__ scores,
                                                            int32_t* __restrict__ ids,
                                                            float* __restrict__ wout,
                                                            int32_t* err) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  select_token<P>(logits, nparts, part_stride, logits_out, t, E, bias, G, TG, K, norm, rsf, scores, ids, wout, err,
                  warp, lane, T > 8);
}

// W (FP32) -> [W1 | W2 | W3] (BF16, side by side along K): W1 = bf16(W),
// W2 = bf16(W - W1), W3 = bf16(W - W1 - W2).  Each difference is exact in FP32
// and each term keeps 8 more significand bits, so sum(x * Wi) with FP32
// accumulation carries FP32-level precision for BF16 x (exact in BF16).
__global__ void split_bf16x3_kernel(const float* __restrict__ w, int E, int d, bf16* __restrict__ out) {
  pdl_wait();
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
cudaError_t launch_select_p(const float* logits, int nparts, int64_t part_stride, float* logits_out, int T, int E,
                            const float* bias, int G, int TG, int K, int norm, float rsf, float* scores, int32_t* ids,
                            float* w, int32_t* err, cudaStream_t s) {
  launch_k(router_select_kernel<P>, (unsigned)ceil_div(T, 8), 256, 0, s, logits, nparts, part_stride, logits_out, T,
           E, bias, G, TG, K, norm, rsf, scores, ids, w, err);
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

// ---------------------------------------------------------------------------
// logits, 33..64 tokens of a wide router (E >= 256): a CTA computes 16 experts x
// TT tokens.  Each 256-wide K chunk of its TT token rows is staged in shared
// memory (FP32) once for all 8 warps; a warp owns 2 experts, a lane 4 + 4
// values of each chunk (k0 + 4l .. +3 and k0 + 128 + 4l .. +3, conflict-free
// 16-byte reads), with 2 x TT FP32 partial sums in registers, added across
// the lanes by a fixed shuffle tree at the end.  The token rows are read from
// L2 once per 16 experts instead of once per 2.
// ---------------------------------------------------------------------------
template <int TT, bool XF32>
__global__ void __launch_bounds__(256) router_logits_wide(const void* __restrict__ X, int T, int d,
                                                          const float* __restrict__ Wr, int E,
                                                          float* __restrict__ logits) {
  pdl_wait();
  constexpr int KC = 256, EW = 2;
  __shared__ __align__(16) float xs[TT][KC];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int eb = blockIdx.x * 16 + warp * EW;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  float acc[EW][TT];
#pragma unroll
  for (int i = 0; i < EW; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[i][t] = 0.f;
  for (int k0 = 0; k0 < d; k0 += KC) {
    __syncthreads();                        // the previous chunk has been read
    for (int i = threadIdx.x; i < TT * KC / 4; i += 256) {
      const int r = i / (KC / 4), c4 = (i % (KC / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < nt && k0 + c4 < d) {
        if (XF32) {
          v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(X) + (int64_t)(t0 + r) * d + k0 + c4);
        } else {
          const uint2 q = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(X) + (int64_t)(t0 + r) * d + k0 + c4);
          v = make_float4(bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y));
        }
      }
      *reinterpret_cast<float4*>(&xs[r][c4]) = v;
    }
    __syncthreads();
    float4 wa[EW], wb[EW];
#pragma unroll
    for (int i = 0; i < EW; ++i) {
      const int e = eb + i;
      wa[i] = wb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < E) {
        const float* w = Wr + (int64_t)e * d + k0;
        if (k0 + 4 * lane < d) wa[i] = ldg_stream_f4(w + 4 * lane);
        if (k0 + 128 + 4 * lane < d) wb[i] = ldg_stream_f4(w + 128 + 4 * lane);
      }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      const float4 xa = *reinterpret_cast<const float4*>(&xs[t][4 * lane]);
      const float4 xb = *reinterpret_cast<const float4*>(&xs[t][128 + 4 * lane]);
#pragma unroll
      for (int i = 0; i < EW; ++i) {
        float a = acc[i][t];
        a = fmaf(wa[i].x, xa.x, a); a = fmaf(wa[i].y, xa.y, a); a = fmaf(wa[i].z, xa.z, a); a = fmaf(wa[i].w, xa.w, a);
        a = fmaf(wb[i].x, xb.x, a); a = fmaf(wb[i].y, xb.y, a); a = fmaf(wb[i].z, xb.z, a); a = fmaf(wb[i].w, xb.w, a);
        acc[i][t] = a;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < EW; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float v = acc[i][t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && t < nt && eb + i < E) logits[(int64_t)(t0 + t) * E + eb + i] = v;
    }
}

template <int TT>
cudaError_t launch_wide(const void* x, int act, int T, int d, const float* w, int E, float* logits, cudaStream_t s) {
  const dim3 grid((unsigned)ceil_div(E, 16), (unsigned)ceil_div(T, TT));
  if (act == MOE_DT_F32)
    launch_k(router_logits_wide<TT, true>, grid, 256, 0, s, x, T, d, w, E, logits);
  else
    launch_k(router_logits_wide<TT, false>, grid, 256, 0, s, x, T, d, w, E, logits);
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
                                 float* logits, cudaStream_t s, void* w_split, float* parts, int* nparts) {
  *nparts = 1;
  if (T <= 0) return cudaSuccess;
  if (w_split && act == MOE_DT_BF16 && T > 64 && E % 32 == 0 && d % 64 == 0) {
    const int64_t n = (int64_t)E * d;
    launch_k(split_bf16x3_kernel, (unsigned)std::min<int64_t>(ceil_div(n, 256), 2048), 256, 0, s, w_router, E, d, reinterpret_cast<bf16*>(w_split));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    GemvArgs a{};
    a.W = w_split; a.N = E; a.K = 3 * d; a.X = x; a.x_ld = d; a.dense_rows = T;
    a.out_ld = E;
    // full 256-row tiles; the K = 3d reduction is split into up to kRouterParts
    // parts when the row x expert tiles alone cannot fill the GPU (the
    // selection kernel adds the parts)
    const int bn = 256;
    int ks = 1;
    if (parts) {
      const int64_t tiles = ceil_div(T, bn) * ceil_div(E, 256);
      ks = (int)std::min<int64_t>(kRouterParts, std::max<int64_t>(1, ceil_div(2 * 152, tiles)));
    }
    a.out = ks > 1 ? parts : logits;
    *nparts = ks;
    return launch_gemm_tc(a, EPI_STORE, true, E, T, 0, bn, s, d, ks);
  }
  if (T <= 4) return launch_small<4>(x, act, T, d, w_router, E, logits, s);
  if (T > 32 && T <= 64 && E >= 256 && d % 8 == 0) {
    // wide routers above 32 tokens: token rows staged once per 16 experts
    // (Super NVFP4 layer at 64 tokens 0.338 -> 0.330 ms; at 8 and 16 tokens
    // the per-2-experts kernel below measured 5-8 us faster)
    return launch_wide<16>(x, act, T, d, w_router, E, logits, s);
  }
  if (T <= 64) return launch_small<8>(x, act, T, d, w_router, E, logits, s);
  dim3 grid((unsigned)ceil_div(T, 64), (unsigned)ceil_div(E, 64));
  if (act == MOE_DT_F32)
    launch_k(router_logits_tiled<true>, grid, 256, 0, s, x, T, d, w_router, E, logits);
  else
    launch_k(router_logits_tiled<false>, grid, 256, 0, s, x, T, d, w_router, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_router_select(const float* logits, int nparts, int64_t part_stride, float* logits_out, int T,
                                 int E, const float* bias, int G, int TG, int K, int norm, float rsf, float* scores,
                                 int32_t* ids, float* w, int32_t* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int P = (int)ceil_div(E, 32);
#define MOE_SELECT(PP) \
  return launch_select_p<PP>(logits, nparts, part_stride, logits_out, T, E, bias, G, TG, K, norm, rsf, scores, ids, w, \
                             err, s)
  if (P <= 1) MOE_SELECT(1);
  if (P <= 2) MOE_SELECT(2);
  if (P <= 4) MOE_SELECT(4);
  if (P <= 8) MOE_SELECT(8);
  if (P <= 16) MOE_SELECT(16);
  MOE_SELECT(32);
#undef MOE_SELECT
}

}  // namespace moe
