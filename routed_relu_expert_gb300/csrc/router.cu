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
// logits, 5..8 and 33..64 tokens of a wide router (E >= 256): a CTA computes
// 8 * EW experts x TT tokens over 256-wide K chunks.  Each chunk's weight rows
// (FP32) and TT token rows (as stored) are copied into shared memory with cp.async, four
// chunks in flight, so the copies of the next three chunks overlap the
// products of the current one.  A warp owns EW experts, a lane 4 + 4 values of
// each chunk (k0 + 4l .. +3 and k0 + 128 + 4l .. +3: conflict-free reads),
// with EW x TT FP32 partial sums in registers, added across the lanes by a
// fixed shuffle tree at the end.  The token rows are read from L2 once per
// 8 * EW experts.
// ---------------------------------------------------------------------------
constexpr int kWideKC = 256, kWideStages = 4;

// one stage: 8 * EW weight rows and TT token rows of one K chunk
template <int TT, int EW, bool XF32>
constexpr int wide_stage_bytes() { return 8 * EW * kWideKC * 4 + TT * kWideKC * (XF32 ? 4 : 2); }

__device__ __forceinline__ void wide_cp16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;     // 0: the 16 bytes are zero-filled, nothing is read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

template <int TT, int EW, bool XF32>
__global__ void __launch_bounds__(256, 1) router_logits_wide(const void* __restrict__ X, int T, int d,
                                                             const float* __restrict__ Wr, int E,
                                                             float* __restrict__ logits) {
  pdl_wait();
  constexpr int KC = kWideKC, EPC = 8 * EW, S = kWideStages;
  constexpr int XB = XF32 ? 4 : 2;                          // bytes of one token value
  constexpr int W_BYTES = EPC * KC * 4, STAGE = wide_stage_bytes<TT, EW, XF32>();
  constexpr int W_PIECES = W_BYTES / 16 / 256;              // 16-byte copies a thread issues per chunk
  constexpr int X_PIECES = (STAGE - W_BYTES) / 16 / 256;
  constexpr int XPR = KC * XB / 16;                         // 16-byte pieces in a chunk of a token row
  static_assert(W_BYTES % (16 * 256) == 0 && (STAGE - W_BYTES) % (16 * 256) == 0, "whole copies per thread");
  extern __shared__ __align__(16) unsigned char wide_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e_blk = blockIdx.x * EPC;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  const int nchunks = (d + KC - 1) / KC;
  const unsigned char* xbytes = reinterpret_cast<const unsigned char*>(X);
  const uint32_t sbase = smem_u32(wide_smem);
  // chunk c into stage c % S: weight rows [e_blk, e_blk + 16) then token rows
  // [t0, t0 + TT), zero past E, the tile's rows or d (d is a multiple of 8)
  auto issue = [&](int c) {
    const uint32_t st = sbase + (uint32_t)((c % S) * STAGE);
    const int k0 = c * KC;
#pragma unroll
    for (int j = 0; j < W_PIECES; ++j) {
      const int i = threadIdx.x + j * 256;
      const int r = i / (KC / 4), k = k0 + (i % (KC / 4)) * 4;
      const bool ok = e_blk + r < E && k < d;
      wide_cp16(st + 16u * i, ok ? (const void*)(Wr + (int64_t)(e_blk + r) * d + k) : (const void*)Wr, ok);
    }
#pragma unroll
    for (int j = 0; j < X_PIECES; ++j) {
      const int i = threadIdx.x + j * 256;
      const int r = i / XPR, k = k0 + (i % XPR) * (16 / XB);
      const bool ok = r < nt && k < d;
      wide_cp16(st + W_BYTES + 16u * i, ok ? (const void*)(xbytes + ((int64_t)(t0 + r) * d + k) * XB) : X, ok);
    }
  };
  float acc[EW][TT];
#pragma unroll
  for (int i = 0; i < EW; ++i)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[i][t] = 0.f;
#pragma unroll
  for (int c = 0; c < S - 1; ++c) {
    if (c < nchunks) issue(c);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int c = 0; c < nchunks; ++c) {
    if (c + S - 1 < nchunks) issue(c + S - 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(S - 1) : "memory");   // this thread's copies of chunk c
    __syncthreads();                                                  // everyone's
    const unsigned char* st = wide_smem + (c % S) * STAGE;
    const float* ws = reinterpret_cast<const float*>(st);
    float4 wa[EW], wb[EW];
#pragma unroll
    for (int i = 0; i < EW; ++i) {
      wa[i] = *reinterpret_cast<const float4*>(ws + (warp * EW + i) * KC + 4 * lane);
      wb[i] = *reinterpret_cast<const float4*>(ws + (warp * EW + i) * KC + 128 + 4 * lane);
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float4 xa, xb;
      if (XF32) {
        const float* xs = reinterpret_cast<const float*>(st + W_BYTES) + t * KC;
        xa = *reinterpret_cast<const float4*>(xs + 4 * lane);
        xb = *reinterpret_cast<const float4*>(xs + 128 + 4 * lane);
      } else {
        const bf16* xs = reinterpret_cast<const bf16*>(st + W_BYTES) + t * KC;
        const uint2 qa = *reinterpret_cast<const uint2*>(xs + 4 * lane);
        const uint2 qb = *reinterpret_cast<const uint2*>(xs + 128 + 4 * lane);
        xa = make_float4(bf16_lo(qa.x), bf16_hi(qa.x), bf16_lo(qa.y), bf16_hi(qa.y));
        xb = make_float4(bf16_lo(qb.x), bf16_hi(qb.x), bf16_lo(qb.y), bf16_hi(qb.y));
      }
#pragma unroll
      for (int i = 0; i < EW; ++i) {
        float a = acc[i][t];
        a = fmaf(wa[i].x, xa.x, a); a = fmaf(wa[i].y, xa.y, a); a = fmaf(wa[i].z, xa.z, a); a = fmaf(wa[i].w, xa.w, a);
        a = fmaf(wb[i].x, xb.x, a); a = fmaf(wb[i].y, xb.y, a); a = fmaf(wb[i].z, xb.z, a); a = fmaf(wb[i].w, xb.w, a);
        acc[i][t] = a;
      }
    }
    __syncthreads();                      // stage c % S is refilled by the next iteration's copies
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  const int eb = e_blk + warp * EW;
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

template <int TT, int EW, bool XF32>
cudaError_t launch_wide_t(const void* x, int T, int d, const float* w, int E, float* logits, cudaStream_t s) {
  auto kernel = router_logits_wide<TT, EW, XF32>;
  constexpr int smem = kWideStages * wide_stage_bytes<TT, EW, XF32>();
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([&](int&) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)ceil_div(E, 8 * EW), (unsigned)ceil_div(T, TT));
  launch_k(kernel, grid, 256, smem, s, x, T, d, w, E, logits);
  return cudaGetLastError();
}

template <int TT, int EW>
cudaError_t launch_wide(const void* x, int act, int T, int d, const float* w, int E, float* logits, cudaStream_t s) {
  if (act == MOE_DT_F32) return launch_wide_t<TT, EW, true>(x, T, d, w, E, logits, s);
  return launch_wide_t<TT, EW, false>(x, T, d, w, E, logits, s);
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
    // wide routers above 32 tokens: weight and token rows copied into shared
    // memory four K chunks ahead (Super NVFP4 layer at 64 tokens 0.293 ->
    // 0.280 ms, at 33 tokens 0.248 -> 0.241; used from 5 tokens on it measured
    // equal at 8 tokens and 1-2 % slower at 16 than the per-2-experts kernel
    // below)
    return launch_wide<16, 2>(x, act, T, d, w_router, E, logits, s);
  }
  if (T > 4 && T <= 8 && E >= 256 && d % 8 == 0) {
    // the same pipeline at 8 experts x 8 tokens a CTA (Super NVFP4 layer at 8
    // tokens 0.146 -> 0.1435 ms, one run).  Measured no faster, or slower, at 9-32
    // tokens of a wide router and at 5-64 tokens of the 128-expert router
    // (Nano at 16 tokens 0.217 -> 0.231 ms: 32 CTAs)
    return launch_wide<8, 1>(x, act, T, d, w_router, E, logits, s);
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
