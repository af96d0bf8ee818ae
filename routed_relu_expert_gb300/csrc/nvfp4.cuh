// NVFP4 decoding helpers (E2M1 values, E4M3 block scales) shared by the
// streaming GEMV and the tensor-core GEMM.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

// the 8 values of one 32-bit word of NVFP4 bytes as 4 FP16 pairs (byte j -> pair j,
// its low nibble in the low half)
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}

// two E4M3 scale bytes (low byte first) as an FP16 pair
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t s16) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)s16));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// FP16 pair -> BF16 pair (exact for the E2M1 x E4M3 products: at most 6
// significant bits, magnitudes 2^-10 .. 2688)
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t v) {
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&v));
  return (uint32_t)bf16_bits(f.x) | ((uint32_t)bf16_bits(f.y) << 16);
}

}  // namespace moe
