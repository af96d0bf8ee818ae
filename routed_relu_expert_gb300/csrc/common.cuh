// Shared device helpers for the routed ReLU^2 MoE kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// Workspace header: first 256 bytes of every workspace.
// ---------------------------------------------------------------------------
struct WsHeader {
  int32_t err;          // device error bits (MOE_DEVERR_*)
  int32_t n_active;     // experts with at least one route (moe_dispatch)
  int32_t n_tiles;      // tensor-core tiles of the current schedule
  int32_t max_rows;     // largest per-expert route count
  int32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

__device__ __forceinline__ void set_error(int32_t* err, int32_t bit) {
  if (err) atomicOr(err, bit);   // integer flag only; no effect on results
}

// ---------------------------------------------------------------------------
// conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  bf16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------
// 16-byte streaming load through the non-coherent path, not kept in L1
// (weights are read once per step).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ float4 ldg_stream_f4(const float* p) {
  const uint4 q = ldg_stream(p);
  return make_float4(__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z), __uint_as_float(q.w));
}

// 16-byte load of reused data (activations): cached normally.
__device__ __forceinline__ uint4 ldg_keep(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------------------
// legacy warp MMA used by the weight-streaming (decode) kernels, where HBM
// bandwidth, not tensor throughput, is the bound:
// D[16x8] += A[16x16] (bf16, row) * B[16x8] (bf16, col), FP32 accumulate.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the same with FP16 operands
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: every kernel of the library is launched so
// that the launch of its successor on the stream is prepared while it runs; a
// kernel waits for its predecessor's results to be complete and visible (wait)
// before reading any of them, a no-op for a kernel launched without the
// attribute.  No kernel releases its successor early
// (griddepcontrol.launch_dependents): blocks released early sit resident,
// waiting, in SM slots that the shared expert on the concurrent stream needs,
// and on GB300 that cost the Super layer 4-56 us a step (T = 1..4096) while
// an early release gained at most 1 us on the single-chain steps.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// shared-memory addresses, the global nanosecond timer (bounded waits) and
// mbarrier operations on this CTA's shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// the same, suspending the thread for at most about `ns` nanoseconds while the
// phase is incomplete (for waits whose wake-up latency is on a critical path:
// the default suspension can outlast the phase by hundreds of nanoseconds)
__device__ __forceinline__ bool mbar_try_ns(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------------------
// small integer helpers
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe
