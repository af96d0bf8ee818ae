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

// true if either BF16 value of the pair is beyond FP16's range (a BF16
// magnitude of at least 65536, infinity or NaN: the BF16 values below it end
// at 65280, inside FP16's 65504)
__device__ __forceinline__ bool bf16x2_beyond_f16(uint32_t v) {
  return (v & 0x7FFFu) >= 0x4780u || ((v >> 16) & 0x7FFFu) >= 0x4780u;
}
__device__ __forceinline__ bool bf16x4_beyond_f16(uint4 q) {
  return bf16x2_beyond_f16(q.x) || bf16x2_beyond_f16(q.y) || bf16x2_beyond_f16(q.z) || bf16x2_beyond_f16(q.w);
}

// BF16 pair -> FP16 pair (exact inside FP16's range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// the 8 values of one 32-bit word of NVFP4 bytes as 4 BF16 pairs (pair j =
// values 2j, 2j+1), exact.  Byte permutes look up the high and the low byte of
// each magnitude's BF16 pattern (0, 0.5, 1, 1.5, 2, 3, 4, 6) from two 8-byte
// tables, interleave them, and move each value's sign bit to bit 15 or 31:
// all full-rate integer operations, no conversion unit.
__device__ __forceinline__ void e2m1x8_to_bf16x2(uint32_t w, uint32_t (&o)[4]) {
  constexpr uint32_t kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;   // high bytes of magnitudes 0-3, 4-7
  constexpr uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u;   // low bytes
  const uint32_t sel = w & 0x77777777u;                       // magnitude index of each nibble
  const uint32_t hi03 = __byte_perm(kHiA, kHiB, sel), hi47 = __byte_perm(kHiA, kHiB, sel >> 16);
  const uint32_t lo03 = __byte_perm(kLoA, kLoB, sel), lo47 = __byte_perm(kLoA, kLoB, sel >> 16);
  o[0] = __byte_perm(lo03, hi03, 0x5140);
  o[1] = __byte_perm(lo03, hi03, 0x7362);
  o[2] = __byte_perm(lo47, hi47, 0x5140);
  o[3] = __byte_perm(lo47, hi47, 0x7362);
  // sign of value 2k: bit 8k+3 (bit 7 of byte k after << 4); of value 2k+1: bit 8k+7
  const uint32_t t = w & 0x88888888u, t4 = t << 4;
  o[0] |= __byte_perm(t4, t, 0x4000) & 0x80008000u;
  o[1] |= __byte_perm(t4, t, 0x5010) & 0x80008000u;
  o[2] |= __byte_perm(t4, t, 0x6020) & 0x80008000u;
  o[3] |= __byte_perm(t4, t, 0x7030) & 0x80008000u;
}

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// FP16 pair -> BF16 pair (exact for the E2M1 x E4M3 products: at most 6
// significant bits, magnitudes 2^-10 .. 2688)
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t v) {
  const float2 f = __half22float2(*reinterpret_cast<__half2*>(&v));
  return (uint32_t)bf16_bits(f.x) | ((uint32_t)bf16_bits(f.y) << 16);
}

}  // namespace moe
