// Output stage shared by the streaming GEMV and the tensor-core grouped GEMM:
// one accumulated value v = sum_k X[row, k] W[f, k] becomes one stored output.
#pragma once

#include "internal.h"

#include <cuda_fp16.h>

namespace moe {

// EPI_ADD residual value at (row, f) in the activation type (0 if none)
template <bool ACT_F32>
__device__ __forceinline__ float residual(const GemvArgs& a, int row, int f) {
  if (!a.res) return 0.f;
  const int64_t i = (int64_t)row * a.res_ld + f;
  return ACT_F32 ? reinterpret_cast<const float*>(a.res)[i]
                 : __bfloat162float(reinterpret_cast<const bf16*>(a.res)[i]);
}

template <int EPI, bool OUT_F32, bool ACT_F32>
__device__ __forceinline__ void epilogue(const GemvArgs& a, int seg, int row, int f, float v) {
  if (a.W_gs) v *= a.W_gs[seg];
  const int64_t o = (int64_t)row * a.out_ld + f;
  float r;
  if (EPI == EPI_RELU2) {
    if (ACT_F32) {
      const float u = fmaxf(v, 0.f);
      r = u * u;
    } else {
      const float u = fmaxf(round_bf16(v), 0.f);
      r = u * u;                    // exact in FP32: product of two 8-bit significands
    }
  } else if (EPI == EPI_SCALE) {
    const int t = a.route_token[row], k = a.route_slot[row];
    r = a.topw[(int64_t)t * a.top_k + k] * v;
  } else if (EPI == EPI_ADD) {
    r = v + (a.add_src ? a.add_src[(int64_t)row * a.add_ld + f] : 0.f);
    r += residual<ACT_F32>(a, row, f);
  } else {
    r = v;
  }
  if (OUT_F32 || ACT_F32) {
    reinterpret_cast<float*>(a.out)[o] = r;
  } else {
    reinterpret_cast<bf16*>(a.out)[o] = __float2bfloat16_rn(r);
  }
}

// The output value before storage, from the per-tensor-scaled accumulation v
// and, for EPI_SCALE, the row's routing weight wr.
template <int EPI, bool ACT_F32>
__device__ __forceinline__ float epi_value(const GemvArgs& a, int row, int f, float v, float wr) {
  if (EPI == EPI_RELU2) {
    const float u = ACT_F32 ? fmaxf(v, 0.f) : fmaxf(round_bf16(v), 0.f);
    return u * u;
  } else if (EPI == EPI_SCALE) {
    return wr * v;
  } else if (EPI == EPI_ADD) {
    const float r = v + (a.add_src ? a.add_src[(int64_t)row * a.add_ld + f] : 0.f);
    return r + residual<ACT_F32>(a, row, f);
  }
  return v;
}

// The same with the segment's per-tensor scale (1 if none) and, for
// EPI_SCALE, the row's routing weight, both fetched earlier by the caller so
// that their load latency overlaps the weight stream.
template <int EPI, bool OUT_F32, bool ACT_F32>
__device__ __forceinline__ void epilogue_pre(const GemvArgs& a, int row, int f, float v, float gs, float wr) {
  const float r = epi_value<EPI, ACT_F32>(a, row, f, v * gs, wr);
  const int64_t o = (int64_t)row * a.out_ld + f;
  if (OUT_F32 || ACT_F32) {
    reinterpret_cast<float*>(a.out)[o] = r;
  } else {
    reinterpret_cast<bf16*>(a.out)[o] = __float2bfloat16_rn(r);
  }
}

// BF16-activation output stored as FP16: the BF16 value itself (exact while
// inside FP16's range), for a consumer that multiplies in FP16.
template <int EPI>
__device__ __forceinline__ void epilogue_pre_f16(const GemvArgs& a, int row, int f, float v, float gs, float wr) {
  const float r = round_bf16(epi_value<EPI, false>(a, row, f, v * gs, wr));
  if (!(fabsf(r) <= 65504.f) && a.err) set_error(a.err, MOE_DEVERR_RANGE);
  reinterpret_cast<__half*>(a.out)[(int64_t)row * a.out_ld + f] = __float2half_rn(r);
}

// routing weight of packed row `row` (EPI_SCALE)
__device__ __forceinline__ float route_weight(const GemvArgs& a, int row) {
  return a.topw[(int64_t)a.route_token[row] * a.top_k + a.route_slot[row]];
}

}  // namespace moe
