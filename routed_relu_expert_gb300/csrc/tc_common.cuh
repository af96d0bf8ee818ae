// Shared pieces of the tensor-core (tcgen05) kernels: PTX wrappers for
// mbarriers, TMA, tcgen05 MMA / commit / TMEM loads, the shared-memory and
// instruction descriptors, the walk over (segment, feature tile, row tile)
// units, the output stage, and the host-side tensor-map encoders.
#pragma once

#include "epilogue.cuh"
#include "nvfp4.cuh"

#include <cuda.h>

#include <mutex>

namespace moe {
namespace tc {

constexpr int BM = 128;                        // features per CTA (TMEM lanes)
constexpr int BK = 64;                         // K per stage: one 128-byte swizzle row
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
// (shared memory addresses, the global timer and the basic mbarrier
// operations are in common.cuh)

// the same with cluster-scope acquire: for barriers the peer CTA arrives on
__device__ __forceinline__ bool mbar_try_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete; false if this thread
// gave up or another role raised the abort flag.  SHORT: suspend for short
// spells only (for the roles whose wake-up latency is on the critical path of
// every stage or tile).
template <bool CL = false, bool SHORT = false>
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  auto probe = [&]() {
    return CL ? mbar_try_cl(bar, parity) : SHORT ? mbar_try_ns(bar, parity, 32u) : mbar_try(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (probe()) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      set_error(err, MOE_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// ---- cluster (CTA pair) helpers ----
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared-memory offset in CTA 0 of the cluster
__device__ __forceinline__ uint32_t map_to_rank0(uint32_t addr) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(addr));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// shared -> global tensor store of one box; completion tracked by bulk groups
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// pair form: the copy lands in this CTA's shared memory and completes its
// bytes on an mbarrier of either CTA of the pair (here: CTA 0's)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int CG>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  if (CG == 2)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` when this thread's MMAs so far are complete; CG 2: on the
// barrier at the same offset in each CTA of `mask`
template <int CG>
__device__ __forceinline__ void tc_commit(uint32_t bar, uint16_t mask = 3) {
  if (CG == 2)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, rows of 128 B,
// 8-row groups 1024 B apart; the tile base is 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);     // start address (16-byte units)
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused by swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: BF16 (or, F16, FP16) A and B (K-major),
// FP32 D, M x N.
__device__ __forceinline__ uint32_t idesc_f16kind(int M, int N, bool F16) {
  const uint32_t fmt = F16 ? 0u : 1u;          // operand format: 0 FP16, 1 BF16
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
struct Tile {
  int seg, m0, row0, rows;
  int kb0, kb1;        // k-blocks [kb0, kb1) of this unit (all of K unless split)
  int orow0;           // first output row (row0 shifted by the unit's K-part slab)
};

// Row-tile prefix over segments: prefix[e] = row tiles of segments < e, each
// segment holding ceil(rows / bn) tiles; prefix[E] = all of them.  Every one of
// the block's nthr threads takes part (it contains a __syncthreads); the
// caller synchronises before reading prefix.  scan_tmp: 32 ints.
__device__ __forceinline__ void row_tile_prefix(const GemvArgs& a, int E, int bn, int nthr, int* scan_tmp,
                                                int* prefix) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (E + nthr - 1) / nthr;
  const int e0 = threadIdx.x * per;
  int local = 0;
  for (int e = e0; e < min(E, e0 + per); ++e) local += (a.offsets[e + 1] - a.offsets[e] + bn - 1) / bn;
  int x = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) scan_tmp[warp] = x;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += scan_tmp[w];
  int run = wbase + x - local;
  for (int e = e0; e < min(E, e0 + per); ++e) {
    prefix[e] = run;
    run += (a.offsets[e + 1] - a.offsets[e] + bn - 1) / bn;
  }
  // (e0 >= E for the last threads: they still write prefix[E] correctly as the block total)
  if (threadIdx.x == nthr - 1) prefix[E] = wbase + x;
}

// unit t -> (K part, row tile, feature tile); parts outermost, so units that
// run together share their K range
// (offs: the segment offsets, a.offsets or a copy of them in shared memory)
__device__ __forceinline__ void decode_tile(int t, const int* prefix, int E, int m_tiles, int tile_m, int bn,
                                            const GemvArgs& a, int per_part, int ksplit, int nkb, Tile& ti,
                                            const int* offs = nullptr) {
  if (!offs) offs = a.offsets;
  const int ks = t / per_part;
  t -= ks * per_part;
  const int q = t / m_tiles, m = t - q * m_tiles;
  int seg = 0, nt = q, base = 0, count = a.dense_rows;
  if (a.offsets) {
    int lo = 0, hi = E;                       // prefix[lo] <= q < prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= q) lo = mid; else hi = mid;
    }
    seg = lo;
    nt = q - prefix[lo];
    base = offs[lo];
    count = offs[lo + 1] - base;
  }
  ti.seg = seg;
  ti.m0 = m * tile_m;
  ti.row0 = base + nt * bn;
  ti.rows = min(bn, count - nt * bn);
  ti.kb0 = (int)((int64_t)ks * nkb / ksplit);
  ti.kb1 = (int)((int64_t)(ks + 1) * nkb / ksplit);
  ti.orow0 = ti.row0 + ks * a.dense_rows;   // K parts: dense products only
}

// Epilogue of 32 accumulator columns (rows row0+c0 .. +31) of one feature f;
// the warp's 32 lanes hold features f0 .. f0+31 (all valid or all beyond N).
// The routing weight of each row (EPI_SCALE) was fetched at the start of the
// tile into `wrow`.  A full chunk of 32 rows is staged in shared memory as
// [row][32 features] and written by one TMA store (a few wide writes instead of
// 32 two- or four-byte stores per thread); a partial chunk, or an output
// without a tensor map, is stored element by element.
// OUT16: BF16-activation output stored as FP16 copies of the BF16 values.
template <int EPI, bool OUT_F32, bool OUT16>
__device__ __forceinline__ void tile_epilogue(const GemvArgs& a, const CUtensorMap* out_map, const Tile& ti, int c0,
                                              int f0, int lane, const float* wrow, uint8_t* stg, float (&v)[32]) {
  constexpr bool F32 = OUT_F32 || EPI == EPI_SCALE;
  const int nc = min(32, ti.rows - c0);
  const int f = f0 + lane;
  if (f0 >= a.N) return;
  if (EPI == EPI_SCALE) {
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] *= wrow[c0 + c];
  }
  if (a.W_gs) {
    const float gs = a.W_gs[ti.seg];
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] *= gs;
  }
  if (EPI == EPI_ADD && a.add_src) {
    float add[32];
#pragma unroll
    for (int c = 0; c < 32; ++c)
      add[c] = c < nc ? a.add_src[(int64_t)(ti.row0 + c0 + c) * a.add_ld + f] : 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] += add[c];
  }
  if (EPI == EPI_ADD && a.res) {
    // BF16 residual rows (the tensor-core path runs BF16 activations only)
    float res[32];
#pragma unroll
    for (int c = 0; c < 32; ++c)
      res[c] = c < nc ? __bfloat162float(reinterpret_cast<const bf16*>(a.res)[(int64_t)(ti.row0 + c0 + c) * a.res_ld + f])
                      : 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] += res[c];
  }
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if (EPI == EPI_RELU2) {
      const float u = fmaxf(round_bf16(v[c]), 0.f);
      v[c] = u * u;
    }
  }
  if (OUT16) {
    // FP16 copies of the BF16 values: a value beyond FP16's range is flagged
    // (rounding is monotonic, so the rounded maximum decides)
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) m = fmaxf(m, c < nc ? fabsf(v[c]) : 0.f);
    if (round_bf16(m) > 65504.f && a.err) set_error(a.err, MOE_DEVERR_RANGE);
  }
  if (out_map && nc == 32) {
    if (lane == 0) bulk_wait_read_all();   // the previous chunk's store has left the staging buffer
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if (F32)
        reinterpret_cast<float*>(stg)[c * 32 + lane] = v[c];
      else if (OUT16)
        reinterpret_cast<__half*>(stg)[c * 32 + lane] = __float2half_rn(round_bf16(v[c]));
      else
        reinterpret_cast<bf16*>(stg)[c * 32 + lane] = __float2bfloat16_rn(v[c]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) tma_store_2d(out_map, smem_u32(stg), f0, ti.orow0 + c0);
    return;
  }
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if (c >= nc) break;
    const int64_t o = (int64_t)(ti.orow0 + c0 + c) * a.out_ld + f;
    if (F32)
      reinterpret_cast<float*>(a.out)[o] = v[c];
    else if (OUT16)
      reinterpret_cast<__half*>(a.out)[o] = __float2half_rn(round_bf16(v[c]));
    else
      reinterpret_cast<bf16*>(a.out)[o] = __float2bfloat16_rn(v[c]);
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld_elems, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld_elems * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// packed NVFP4 weights [rows, k / 2] bytes: boxes of 128 rows x 32 bytes (64 values)
inline bool make_packed_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t k) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
  cuuint32_t box[2] = {BK / 2, BM};
  cuuint32_t el[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, el,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// output map for the epilogue's TMA stores; false (element stores instead) if
// the output's base or row pitch is not 16-byte aligned
inline bool make_out_map(CUtensorMap* m, const void* ptr, int64_t rows, int n, int64_t ld, bool f32) {
  EncodeTiledFn fn = encode_fn();
  const int es = f32 ? 4 : 2;
  if (!fn || !ptr || (reinterpret_cast<uintptr_t>(ptr) & 15) || (ld * es) % 16 || n % 32) return false;
  cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t el[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
            strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace tc
}  // namespace moe
