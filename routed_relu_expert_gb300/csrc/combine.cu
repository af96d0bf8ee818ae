// Combine: y_r[t] = sum of token t's routed rows u[row] in ascending expert id,
// FP32, one fixed order (page "NemotronH (Nemotron 3.5 Lightning, Bolt, Super
// VL)", section "Arithmetic": the weighted sum in fp32 in ascending expert id;
// page "Nemotron-3.5-Super 120B on an 8 GB GPU", section "How we know it's
// right": a per-(token, expert) buffer summed in a fixed order instead of
// atomics).  Packed rows are expert-contiguous, so ascending packed row is
// ascending expert id.
#include "internal.h"

#include <algorithm>
#include <climits>

namespace moe {

namespace {

// four consecutive activation values (f32 or bf16) from element i (a multiple of 4)
template <bool ACT_F32>
__device__ __forceinline__ float4 load_act4(const void* p, int64_t i) {
  if (ACT_F32) return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
  const uint2 b = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(p) + i);
  return make_float4(bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y));
}

// grid (T, column blocks of 128 float4s): each thread owns one float4 column of
// one token and loads all of that column's routed rows before adding them in
// row order, so a token's K loads are in flight together
constexpr int kCombineThreads = 128;

template <bool ACT_F32>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ u,
                                                                  const int32_t* __restrict__ tsr, int K, int de,
                                                                  float* y_r, void* y_act,
                                                                  const float* __restrict__ add, const void* res) {
  pdl_wait();
  __shared__ int rows[32];
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    const int r = tsr[(int64_t)t * K + threadIdx.x];
    // rank among the token's rows (rows are distinct; invalid = -1 sorts last)
    const unsigned key = r < 0 ? UINT_MAX : (unsigned)r;
    int rank = 0;
    for (int j = 0; j < K; ++j) {
      const int rj = tsr[(int64_t)t * K + j];
      const unsigned kj = rj < 0 ? UINT_MAX : (unsigned)rj;
      rank += (kj < key) || (kj == key && j < (int)threadIdx.x);
    }
    rows[rank] = r;
  }
  const int nv = de / 4;
  const int v = blockIdx.y * kCombineThreads + threadIdx.x;
  float4 extra = make_float4(0.f, 0.f, 0.f, 0.f);
  if (add && v < nv) extra = reinterpret_cast<const float4*>(add + (int64_t)t * de)[v];
  __syncthreads();
  if (v >= nv) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int B = 8;                   // rows loaded ahead of their adds
  for (int i0 = 0; i0 < K; i0 += B) {
    float4 q[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int r = i0 + i < K ? rows[i0 + i] : -1;
      q[i] = r >= 0 ? reinterpret_cast<const float4*>(u + (int64_t)r * de)[v] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < B; ++i) {
      if (i0 + i < K && rows[i0 + i] >= 0) {
        acc.x += q[i].x; acc.y += q[i].y; acc.z += q[i].z; acc.w += q[i].w;
      }
    }
  }
  if (y_r) reinterpret_cast<float4*>(y_r + (int64_t)t * de)[v] = acc;
  if (add) {
    // output = routed sum + an FP32 term (the shared expert), then one rounding
    acc.x += extra.x; acc.y += extra.y; acc.z += extra.z; acc.w += extra.w;
  }
  if (res) {
    // + the residual row (read before y_act, which may be the same row, is written)
    const float4 q = load_act4<ACT_F32>(res, (int64_t)t * de + 4 * (int64_t)v);
    acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
  }
  if (y_act) {
    if (ACT_F32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(y_act) + (int64_t)t * de)[v] = acc;
    } else {
      uint2 p;
      p.x = (uint32_t)bf16_bits(acc.x) | ((uint32_t)bf16_bits(acc.y) << 16);
      p.y = (uint32_t)bf16_bits(acc.z) | ((uint32_t)bf16_bits(acc.w) << 16);
      reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(y_act) + (int64_t)t * de)[v] = p;
    }
  }
}

template <bool ACT_F32>
__global__ void cast_kernel(const float* __restrict__ src, int64_t n4, void* dst, const void* res) {
  pdl_wait();
  for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < n4; v += (int64_t)gridDim.x * blockDim.x) {
    float4 q = reinterpret_cast<const float4*>(src)[v];
    if (res) {
      const float4 r = load_act4<ACT_F32>(res, 4 * v);
      q.x += r.x; q.y += r.y; q.z += r.z; q.w += r.w;
    }
    if (ACT_F32) {
      reinterpret_cast<float4*>(dst)[v] = q;
    } else {
      uint2 p;
      p.x = (uint32_t)bf16_bits(q.x) | ((uint32_t)bf16_bits(q.y) << 16);
      p.y = (uint32_t)bf16_bits(q.z) | ((uint32_t)bf16_bits(q.w) << 16);
      reinterpret_cast<uint2*>(dst)[v] = p;
    }
  }
}

}  // namespace

cudaError_t launch_cast(const float* src, int64_t n, void* dst, int act, cudaStream_t s, const void* res) {
  if (n <= 0) return cudaSuccess;
  const int64_t n4 = n / 4;
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(n4, 256), 4096);
  if (act == MOE_DT_F32)
    launch_k(cast_kernel<true>, grid, 256, 0, s, src, n4, dst, res);
  else
    launch_k(cast_kernel<false>, grid, 256, 0, s, src, n4, dst, res);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* u, const int32_t* token_slot_row, int T, int K, int de, float* y_r,
                           void* y_act, int act, cudaStream_t s, const float* add, const void* res) {
  if (T <= 0) return cudaSuccess;
  const dim3 grid((unsigned)T, (unsigned)ceil_div(de / 4, kCombineThreads));
  if (act == MOE_DT_F32)
    launch_k(combine_kernel<true>, grid, kCombineThreads, 0, s, u, token_slot_row, K, de, y_r, y_act, add, res);
  else
    launch_k(combine_kernel<false>, grid, kCombineThreads, 0, s, u, token_slot_row, K, de, y_r, y_act, add, res);
  return cudaGetLastError();
}

}  // namespace moe
