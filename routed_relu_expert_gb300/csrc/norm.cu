// RMSNorm prologue of the MoE block (page "Nemotron Is Not One Circuit: Mamba,
// Attention, and MoE Routing", section "The Four Layer Kinds CKE Must
// Preserve": an MoE layer runs RMSNorm, the router, the group-limited top-k,
// the routed ReLU^2 experts plus the shared expert, then the residual add).
//
// xn[t, j] = act(gamma[j] * (x[t, j] * r_t)),  r_t = 1 / sqrt(mean_j(x[t, j]^2) + eps)
//
// all in FP32, one rounding to the activation type at the end.  One CTA per
// token row; each thread's partial sum of squares runs over a fixed set of
// columns, and the partials meet in a fixed tree, so the result does not
// depend on scheduling.  The same kernel clears the workspace header, which
// puts the step's first write of the header in its first kernel.
#include "internal.h"

namespace moe {

namespace {

constexpr int kNormThreads = 256;

template <bool ACT_F32>
__device__ __forceinline__ void load8(const void* x, int64_t i, float (&v)[8]) {
  if (ACT_F32) {
    const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + i);
    const float4 b = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + i + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 q = *reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(x) + i);
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
    v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
  }
}

template <bool ACT_F32>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const void* __restrict__ x,
                                                               const float* __restrict__ gamma, float eps, int d,
                                                               void* __restrict__ xn, uint32_t* __restrict__ hdr,
                                                               int hdr_words) {
  pdl_wait();
  __shared__ float part[kNormThreads / 32];
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < hdr_words; i += kNormThreads) hdr[i] = 0u;
  const int t = blockIdx.x;
  const int64_t row = (int64_t)t * d;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // sum of squares: thread i takes the 8-column chunks i, i + 256, ... in order
  float ss = 0.f;
  for (int j = threadIdx.x * 8; j < d; j += kNormThreads * 8) {
    float v[8];
    load8<ACT_F32>(x, row + j, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane == 0) part[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += part[w];   // the same order in every thread
  const float r = 1.0f / sqrtf(tot / (float)d + eps);
  for (int j = threadIdx.x * 8; j < d; j += kNormThreads * 8) {
    float v[8];
    load8<ACT_F32>(x, row + j, v);
    const float4 g0 = *reinterpret_cast<const float4*>(gamma + j);
    const float4 g1 = *reinterpret_cast<const float4*>(gamma + j + 4);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = g[i] * (v[i] * r);
    if (ACT_F32) {
      float* o = reinterpret_cast<float*>(xn) + row + j;
      *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(o + 4) = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint4 p;
      p.x = (uint32_t)bf16_bits(v[0]) | ((uint32_t)bf16_bits(v[1]) << 16);
      p.y = (uint32_t)bf16_bits(v[2]) | ((uint32_t)bf16_bits(v[3]) << 16);
      p.z = (uint32_t)bf16_bits(v[4]) | ((uint32_t)bf16_bits(v[5]) << 16);
      p.w = (uint32_t)bf16_bits(v[6]) | ((uint32_t)bf16_bits(v[7]) << 16);
      *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(xn) + row + j) = p;
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const void* x, const float* gamma, float eps, int T, int d, int act, void* xn,
                           void* hdr, int hdr_bytes, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (d % 8 || hdr_bytes % 4) return cudaErrorInvalidValue;
  uint32_t* h = reinterpret_cast<uint32_t*>(hdr);
  if (act == MOE_DT_F32)
    launch_k(rmsnorm_kernel<true>, (unsigned)T, kNormThreads, 0, s, x, gamma, eps, d, xn, h, hdr_bytes / 4);
  else
    launch_k(rmsnorm_kernel<false>, (unsigned)T, kNormThreads, 0, s, x, gamma, eps, d, xn, h, hdr_bytes / 4);
  return cudaGetLastError();
}

}  // namespace moe
