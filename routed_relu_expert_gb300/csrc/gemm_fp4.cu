// NVFP4 expert products on the FP4 tensor path.
//
// The weights are NVFP4 (E2M1 values, one E4M3 scale per 16 consecutive K
// values, one FP32 scale per tensor: page "Nemotron-3.5-Super 120B on an 8 GB
// GPU", section "The engine, step by step", item 4).  The block-scaled MMA
// (tcgen05.mma kind::mxf4nvf4, scale_vec::4X) multiplies two NVFP4 operands
// and applies both operands' E4M3 block scales itself, so the weights go from
// HBM to shared memory by TMA and into the MMA without any decoding.  The
// activations are brought into the same format as a sum of NVFP4 terms:
//
//   quant_terms_kernel   a row x (BF16 values) -> g = amax(x) / (6 * 448);
//                        term j of a 16-value block: scale = E4M3_rn(amax(r) /
//                        (6 g)), s = scale * g, code = E2M1_rn(r * (1/s)),
//                        r -= code * s  (r = x before the first term)
//   fp4_gemm_kernel      D[f, row] = sum_j sum_k W[f, k] x_j[row, k] (FP32 in
//                        TMEM), one MMA per term and 64-wide K step into the
//                        same accumulator; out = epilogue(D * g_row * gs_seg)
//
// Kernel layout (one CTA per SM, persistent over (segment, 128-feature tile,
// row tile) units): warp 0 streams the weight tiles with TMA, warp 6 the
// activation terms (every term in one box) and warp 11 their block scales
// (one box issued per thread and stage: an issuing thread manages about one
// box per few hundred cycles), warp 1 issues the MMAs, warps 2-5
// run the epilogue from TMEM (two accumulators, so a tile's epilogue overlaps
// the next tile's MMAs), warps 7-10 place the block scales in TMEM where the
// MMA reads them: row m of the weight tile at (lane m, column c + m / 32), row
// n of the activation tile at (lane 32q + n % 32, column c + n / 32) in every
// lane quarter q (the layout measured on this GPU).  The weight scales come
// straight from global memory (their rows need not be 16-byte aligned), a few
// stages ahead.  Every mbarrier wait is bounded; on expiry the CTA sets
// MOE_DEVERR_TIMEOUT, stops every role, waits (bounded) for its copies and
// MMAs in flight, frees its TMEM and returns.
#include "tc_common.cuh"

#include <algorithm>
#include <cstring>
#include <mutex>

namespace moe {

namespace {

using namespace tc;

constexpr int FP4_K_STAGE = 256;                       // K values per stage (128 bytes a row)
constexpr int ROW_BYTES = FP4_K_STAGE / 2;
constexpr int A_STAGE_BYTES = BM * ROW_BYTES;          // 16 KB
constexpr int kFp4Threads = 384;                       // 12 warps
constexpr int kBWarpF = 6;
constexpr int kSfWarp0 = 7;                            // warps 7..10
constexpr int kSfbWarp = 11;
constexpr int N_HEIGHTS = 4;                           // B boxes of 16, 32, 48, 64 rows
constexpr int kSfPrefetch = 6;                         // weight-scale stages fetched ahead
constexpr size_t kSmemLimit = 227 * 1024;
constexpr int kTileTable = 512;                        // units a CTA finds decoded in shared memory

template <int BNMAX, int NT>
struct Fp4Cfg {
  static constexpr int B_TERM = BNMAX * ROW_BYTES;                       // one term's row tile
  static constexpr int SFB_TERM = BNMAX * 16;                            // its scales for one stage
  static constexpr int STAGE = (A_STAGE_BYTES + NT * (B_TERM + SFB_TERM) + 1023) / 1024 * 1024;
  // 16-row tiles (decode): two CTAs per SM, each with half of TMEM and of
  // shared memory, so two independent pipelines share the SM's tensor core
  // and copy engine (one CTA's single MMA thread waits and issues serially)
  static constexpr int CPS = BNMAX <= 16 ? 2 : 1;
  static constexpr int TMEM_COLS = 512 / CPS;
  // epilogue chunk staged for a TMA store (FP32 at most); tiles of fewer than
  // 32 rows never fill one
  static constexpr int STG = BNMAX >= 32 ? 32 * 32 * 4 : 0;
  static constexpr int EPI_WARP = STG + 2 * BNMAX * 4;                   // + routing weights, row scales
  // MERGE: the terms' rows, stacked, are one B operand of NT * rows, so each
  // K step is one MMA (a block-scaled MMA costs nearly as much for 32 columns
  // as for 192) and the epilogue adds the terms' columns; else one MMA per
  // term into the same accumulator
  static constexpr bool MERGE = NT * BNMAX <= 192;
  static constexpr int ACC_COLS = MERGE ? NT * BNMAX : BNMAX;            // one accumulator
  // every scale-factor address the MMA gets is a multiple of four columns
  static constexpr int SFB_ROW_CHUNKS = (NT * BNMAX + 31) / 32;          // 32-row chunks of stacked rows
  static constexpr int SFB_STEP = MERGE ? (SFB_ROW_CHUNKS <= 4 ? 4 : 8) : 4;   // B scale columns a K step
  static constexpr int SF_COLS = 16 + (MERGE ? 4 * SFB_STEP : 16 * NT);  // TMEM scale columns per slot
  static constexpr int TMEM_SF0 = 2 * ACC_COLS;                          // after the two accumulators
  static_assert(!MERGE || SFB_ROW_CHUNKS <= 8, "merged terms fit eight scale columns");
  static_assert(!MERGE || A_STAGE_BYTES + NT * B_TERM + 32 * SFB_ROW_CHUNKS * 16 <= STAGE,
                "the scale writers' reads stay inside the stage");
  static_assert(ACC_COLS % 4 == 0 && SF_COLS % 16 == 0, "scale and accumulator columns stay aligned");
  static constexpr size_t fixed_smem(int E) {
    return 1024 + (size_t)4 * EPI_WARP + 512 + (16 + 2 * ((size_t)E + 1)) * 4 + 64 + kTileTable * 8;
  }
  static constexpr size_t SMEM_LIMIT = CPS == 1 ? kSmemLimit : 113 * 1024;
  static constexpr int stages_for() {
    int s = 8;
    while (s > 2 && (size_t)s * STAGE + fixed_smem(1024) > SMEM_LIMIT) --s;
    return s;
  }
  static constexpr int STAGES = stages_for();
  // TMEM scale slots: one per stage when they fit, else fewer, reused in turn
  // (DECOUPLED: a slot is rewritten only after the MMAs that read it completed)
  static constexpr int SF_SLOTS =
      (TMEM_COLS - TMEM_SF0) / SF_COLS < STAGES ? (TMEM_COLS - TMEM_SF0) / SF_COLS : STAGES;
  static constexpr bool DECOUPLED = SF_SLOTS < STAGES;
  static_assert((size_t)STAGES * STAGE + fixed_smem(1024) <= SMEM_LIMIT, "shared memory");
  static_assert(SF_SLOTS >= 2 && TMEM_SF0 + SF_SLOTS * SF_COLS <= TMEM_COLS, "tensor memory");
  static_assert(B_TERM % 1024 == 0, "term tiles start on 1024-byte boundaries");
};

struct Fp4Maps {
  CUtensorMap a;                     // packed weights, boxes of 128 rows x 128 bytes
  CUtensorMap b[N_HEIGHTS];          // packed activation terms [terms][rows][K/2]: boxes of
                                     // every term x 16 (i + 1) rows x 128 bytes
  CUtensorMap sfb[N_HEIGHTS];        // their block scales: every term x 16 (i + 1) rows x 16 bytes
  CUtensorMap out;                   // output, boxes of 32 rows x 32 features
};

// The units a CTA visits (t = first, first + step, ...) in increasing order,
// so the segment of the next unit is found by stepping forward from the last
// one instead of a binary search (a single thread's dependent shared-memory
// loads cost about a microsecond per tile otherwise).  Segment e holds row
// tiles [prefix[e], prefix[e + 1]); units are (row tile, feature tile) with
// the feature tile fastest.
struct TileWalk {
  const int* prefix;
  const int* offs;
  int E, m_tiles, bn, dense_rows;
  int seg = -1;
  __device__ __forceinline__ void at(int t, Tile& ti) {
    const int q = t / m_tiles;
    ti.m0 = (t - q * m_tiles) * BM;
    int base, count, nt;
    if (offs) {
      if (seg < 0) {                       // first unit: binary search, prefix[lo] <= q < prefix[hi]
        int lo = 0, hi = E;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (prefix[mid] <= q) lo = mid; else hi = mid;
        }
        seg = lo;
      }
      while (seg + 1 < E && prefix[seg + 1] <= q) ++seg;
      nt = q - prefix[seg];
      base = offs[seg];
      count = offs[seg + 1] - base;
    } else {
      nt = q;
      base = 0;
      count = dense_rows;
    }
    ti.seg = offs ? seg : 0;
    ti.row0 = base + nt * bn;
    ti.rows = min(bn, count - nt * bn);
    ti.orow0 = ti.row0;
    ti.kb0 = 0;
    ti.kb1 = 0;
  }
};

// ---- PTX wrappers for the block-scaled MMA and TMEM stores ----
// kind::mxf4nvf4 instruction descriptor: E2M1 A and B (format 1), both
// K-major, N >> 3, E4M3 block scales (scale format 0), M >> 4
__device__ __forceinline__ uint32_t idesc_mxf4nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st_x2(uint32_t taddr, uint32_t v0, uint32_t v1) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(v0), "r"(v1) : "memory");
}
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3,
                                           uint32_t v4, uint32_t v5, uint32_t v6, uint32_t v7) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(v0),
               "r"(v1), "r"(v2), "r"(v3), "r"(v4), "r"(v5), "r"(v6), "r"(v7)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 8-byte read-only load
__device__ __forceinline__ uint2 ldg_u2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// activation terms
// ---------------------------------------------------------------------------
// E4M3 code of v >= 0 (round to nearest even, saturating at 448)
__device__ __forceinline__ uint32_t e4m3_code(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}
// value of an E4M3 code (exact)
__device__ __forceinline__ float e4m3_val(uint32_t code) {
  const uint32_t h = e4m3x2_to_f16x2(code);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}
// E2M1 codes of (lo, hi) in one byte (lo in the low nibble; round to nearest
// even, saturating at 6) and the two values they stand for
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi, float& qlo, float& qhi) {
  uint16_t b;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n mov.b16 %0, {t, 0};\n}" : "=h"(b) : "f"(hi), "f"(lo));
  uint32_t h;
  asm("{\n .reg .b8 t, t1;\n mov.b16 {t, t1}, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h) : "h"(b));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h);
  qlo = __low2float(hv);
  qhi = __high2float(hv);
  return b & 0xFFu;
}

template <int NT>
__global__ void __launch_bounds__(256) quant_terms_kernel(const bf16* __restrict__ x, int64_t x_ld,
                                                          const int32_t* __restrict__ gather,
                                                          const int32_t* __restrict__ count, int R, int K,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                          float* __restrict__ g, int64_t rows_cap,
                                                          int64_t sf_ld) {
  pdl_wait();
  const int rows = count ? min(*count, R) : R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = K / 16;
  for (int r = blockIdx.x * 8 + warp; r < rows; r += gridDim.x * 8) {
    const int64_t src = gather ? (int64_t)gather[r] : (int64_t)r;
    const bf16* xr = x + src * x_ld;
    // the row's largest magnitude (non-negative floats order as their bits)
    uint32_t am = 0;
    for (int b = lane; b < nb; b += 32) {
      const uint4 v0 = ldg_keep(xr + 16 * b), v1 = ldg_keep(xr + 16 * b + 8);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        am = max(am, __float_as_uint(fabsf(bf16_lo(w[i]))));
        am = max(am, __float_as_uint(fabsf(bf16_hi(w[i]))));
      }
    }
    am = __reduce_max_sync(0xffffffffu, am);
    float gr = __fdiv_rn(__uint_as_float(am), 2688.f);
    if (!(gr > 0.f)) gr = 1.f;
    const float six_g = __fmul_rn(6.f, gr);
    if (lane == 0) g[r] = gr;
    for (int b = lane; b < nb; b += 32) {
      const uint4 v0 = ldg_keep(xr + 16 * b), v1 = ldg_keep(xr + 16 * b + 8);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float amb = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amb = fmaxf(amb, fabsf(v[i]));
        const uint32_t sc = e4m3_code(__fdiv_rn(amb, six_g));
        const float s = __fmul_rn(e4m3_val(sc), gr);
        const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float q0, q1;
          const uint32_t byte = e2m1_pair(__fmul_rn(v[i], inv), __fmul_rn(v[i + 1], inv), q0, q1);
          packed[i >> 3] |= byte << (8 * ((i >> 1) & 3));
          v[i] = __fsub_rn(v[i], __fmul_rn(q0, s));
          v[i + 1] = __fsub_rn(v[i + 1], __fmul_rn(q1, s));
        }
        const int64_t row = (int64_t)j * rows_cap + r;
        *reinterpret_cast<uint2*>(q + row * (K / 2) + 8 * b) = make_uint2(packed[0], packed[1]);
        sf[row * sf_ld + b] = (uint8_t)sc;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the FP4 grouped GEMM
// ---------------------------------------------------------------------------
template <int EPI, bool OUT_F32, int BNMAX, int NT>
__global__ void __launch_bounds__(kFp4Threads, Fp4Cfg<BNMAX, NT>::CPS)
    fp4_gemm_kernel(const __grid_constant__ Fp4Maps maps, const GemvArgs a, int E, int m_tiles, int bn,
                    int tma_out) {
  using C = Fp4Cfg<BNMAX, NT>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint8_t* epi_smem = gbase + STAGES * C::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_smem + 4 * C::EPI_WARP);
  const uint32_t bar0 = smem_u32(bars);
  // afull: a stage's weight tile landed; bfull: its activation terms and their
  // scales landed (from L2, usually well before the weights); sf: the scale
  // writers have placed the stage's scales in TMEM; empty: its MMAs completed
  constexpr int SLOTS = C::SF_SLOTS;
  auto afull_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto bfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  auto sf_bar = [&](int k) { return bar0 + 8u * (3 * STAGES + k); };               // slot k written
  auto sffree_bar = [&](int k) { return bar0 + 8u * (3 * STAGES + SLOTS + k); };   // slot k read
  auto tfull_bar = [&](int i) { return bar0 + 8u * (3 * STAGES + 2 * SLOTS + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (3 * STAGES + 2 * SLOTS + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (3 * STAGES + 2 * SLOTS + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 2 * SLOTS + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* scan_tmp = reinterpret_cast<int*>(tmem_holder + 4);          // [16]
  int* prefix = scan_tmp + 16;                                         // [E+1]
  int* offs = prefix + E + 1;                                          // [E+1] copy of a.offsets
  uint2* table = reinterpret_cast<uint2*>(offs + E + 1);              // [kTileTable] decoded units (prefix is
                                                                       // 8-byte aligned, 2(E+1) ints before)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x, n_units = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(afull_bar(s), 1);
      mbar_init(bfull_bar(s), 2);       // the activation terms and their scales
      mbar_init(empty_bar(s), 1);
    }
    for (int k = 0; k < SLOTS; ++k) {
      mbar_init(sf_bar(k), 128);        // the four scale-writer warps
      mbar_init(sffree_bar(k), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pdl_wait();
  if (a.offsets) {
    for (int e = threadIdx.x; e <= E; e += kFp4Threads) offs[e] = a.offsets[e];
    row_tile_prefix(a, E, bn, kFp4Threads, scan_tmp, prefix);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int total_q = a.offsets ? prefix[E] : (a.dense_rows + bn - 1) / bn;
  const uint32_t tmem_base = *tmem_holder;
  const int total = total_q * m_tiles;
  const int K = a.K;
  const int nkb = (K + FP4_K_STAGE - 1) / FP4_K_STAGE;
  const int64_t rows_cap = a.x_rows_cap;
  TileWalk walk{prefix, a.offsets ? offs : nullptr, E, m_tiles, bn, a.dense_rows};
  // this CTA's first kTileTable units decoded once, in parallel: the roles'
  // single threads then find a unit with one shared-memory load instead of a
  // chain of dependent ones
  const int my_units = total > unit ? (total - unit + n_units - 1) / n_units : 0;
  for (int k = threadIdx.x; k < min(my_units, kTileTable); k += kFp4Threads) {
    TileWalk w = walk;
    Tile tk;
    w.at(unit + k * n_units, tk);
    table[k] = make_uint2((uint32_t)tk.row0,
                          ((uint32_t)tk.seg << 20) | ((uint32_t)(tk.m0 / BM) << 8) | (uint32_t)tk.rows);
  }
  __syncthreads();
  auto tile_of = [&](int k, int t, TileWalk& wk, Tile& ti) {
    if (k < kTileTable) {
      const uint2 e = table[k];
      ti.row0 = ti.orow0 = (int)e.x;
      ti.seg = (int)(e.y >> 20);
      ti.m0 = (int)((e.y >> 8) & 0xFFFu) * BM;
      ti.rows = (int)(e.y & 0xFFu);
      ti.kb0 = ti.kb1 = 0;
    } else {
      wk.at(t, ti);
    }
  };

  if (warp == 0 || warp == kBWarpF || warp == kSfbWarp) {
    const int role = warp == 0 ? 0 : warp == kBWarpF ? 1 : 2;
    const bool is_a = role == 0;
    if (lane == 0) {
      // ------- TMA producers, one box a stage each (an issuing thread manages
      // about one box per few hundred cycles): warp 0 the weight tile, warp 6
      // the activation terms, warp 11 their block scales -------
      int pend[STAGES];
      for (int s = 0; s < STAGES; ++s) pend[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = unit; t < total && ok; t += n_units) {
        Tile ti;
        tile_of((t - unit) / n_units, t, walk, ti);
        const int r16 = (ti.rows + 15) & ~15;
        const int hi = r16 / 16 - 1;
        const uint32_t tx = role == 0 ? (uint32_t)A_STAGE_BYTES
                                      : (uint32_t)(NT * r16 * (role == 1 ? ROW_BYTES : 16));
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait<false, true>(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
          const uint32_t fb = is_a ? afull_bar(stage) : bfull_bar(stage);
          mbar_expect_tx(fb, tx);
          const uint32_t st = base + stage * C::STAGE;
          if (role == 0)
            tma_load_2d(st, &maps.a, kb * ROW_BYTES, ti.seg * a.N + ti.m0, fb);
          else if (role == 1)   // term j's rows land at j * r16 * 128 bytes
            tma_load_3d(st + A_STAGE_BYTES, &maps.b[hi], kb * ROW_BYTES, ti.row0, 0, fb);
          else                  // their scales at j * r16 * 16 bytes
            tma_load_3d(st + A_STAGE_BYTES + NT * C::B_TERM, &maps.sfb[hi], kb * 16, ti.row0, 0, fb);
          pend[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s) {
          if (pend[s] < 0) continue;
          const uint32_t fb = is_a ? afull_bar(s) : bfull_bar(s);
          const uint64_t t0 = globaltimer();
          while (!mbar_try(fb, (uint32_t)pend[s]) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, acc = 0, slot = 0;
      uint32_t phase = 0, acc_phase = 0, sphase = 0;
      bool ok = true, issued = false;
      for (int t = unit; t < total && ok; t += n_units) {
        Tile ti;
        tile_of((t - unit) / n_units, t, walk, ti);
        const int r16 = (ti.rows + 15) & ~15;
        const uint32_t idesc = idesc_mxf4nvf4(BM, C::MERGE ? NT * r16 : r16);
        if (!mbar_wait<false, true>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * C::ACC_COLS);
        uint32_t accumulate = 0;
        for (int kb = 0; kb < nkb; ++kb) {
          // (the scale writers arrive only after seeing the activation copies land)
          if (!mbar_wait<false, true>(sf_bar(slot), sphase, abort_flag, a.err)) { ok = false; break; }
          if (!mbar_wait<false, true>(afull_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = base + stage * C::STAGE;
          const uint32_t sf0 = tmem_base + (uint32_t)(C::TMEM_SF0 + slot * C::SF_COLS);
          const int steps = min(4, (K - kb * FP4_K_STAGE) / 64);
          const uint64_t da = smem_desc_sw128(st);
          const uint64_t db0 = smem_desc_sw128(st + A_STAGE_BYTES);
          for (int s = 0; s < steps; ++s) {
            if constexpr (C::MERGE) {
              mma_fp4(d, da + 2u * s, db0 + 2u * s, idesc, sf0 + 4u * s, sf0 + 16u + (uint32_t)(C::SFB_STEP * s),
                      accumulate);
              accumulate = 1;
            } else {
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                // term j's rows start at j * r16 * 128 bytes (a multiple of 2048)
                const uint64_t db = db0 + (uint64_t)((j * r16 * ROW_BYTES) >> 4);
                mma_fp4(d, da + 2u * s, db + 2u * s, idesc, sf0 + 4u * s, sf0 + 16u + 16u * j + 4u * s, accumulate);
                accumulate = 1;
              }
            }
          }
          issued = true;
          tc_commit<1>(empty_bar(stage));
          if constexpr (C::DECOUPLED) tc_commit<1>(sffree_bar(slot));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (++slot == SLOTS) { slot = 0; sphase ^= 1u; }
        }
        if (!ok) break;
        tc_commit<1>(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && issued) {
        tc_commit<1>(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try(drain_bar, 0u) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp >= kSfWarp0 && warp < kSfWarp0 + 4) {
    // ------- scale writers: warps 7..10, TMEM lane quarter q = warp % 4 -------
    const int q = warp & 3;
    const uint32_t lane_base = tmem_base + ((uint32_t)(32 * q) << 16);
    const int sf_row_bytes = K / 16;
    // the weight scales of this lane's tile row (feature 32q + lane) for one
    // stage: 16 bytes, 4 per 64-wide K step (zero past the end of K)
    int ft = unit, fkb = 0;
    Tile fti;
    TileWalk fwalk = walk;
    if (ft < total) tile_of((ft - unit) / n_units, ft, fwalk, fti);
    auto fetch = [&]() -> uint4 {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (ft >= total) return v;
      const int f = fti.m0 + 32 * q + lane;
      if (f < a.N) {
        const uint8_t* p = a.W_sf + ((int64_t)fti.seg * a.N + f) * sf_row_bytes + fkb * 16;
        const int valid = sf_row_bytes - fkb * 16;             // a multiple of 4
        if (valid >= 8) { const uint2 u = ldg_u2(p); v.x = u.x; v.y = u.y; }
        else if (valid >= 4) v.x = *reinterpret_cast<const uint32_t*>(p);
        if (valid >= 16) { const uint2 u = ldg_u2(p + 8); v.z = u.x; v.w = u.y; }
        else if (valid >= 12) v.z = *reinterpret_cast<const uint32_t*>(p + 8);
      }
      if (++fkb == nkb) {
        fkb = 0;
        ft += n_units;
        if (ft < total) tile_of((ft - unit) / n_units, ft, fwalk, fti);
      }
      return v;
    };
    uint4 ring[kSfPrefetch];
#pragma unroll
    for (int i = 0; i < kSfPrefetch; ++i) ring[i] = fetch();
    int stage = 0, slot = 0, g = 0;
    uint32_t phase = 0, sphase = 0;
    bool ok = true;
    for (int t = unit; t < total && ok; t += n_units) {
      Tile ti;
      tile_of((t - unit) / n_units, t, walk, ti);
      const int r16 = (ti.rows + 15) & ~15;
      for (int kb = 0; kb < nkb; ++kb) {
        const uint4 wa = ring[0];
#pragma unroll
        for (int i = 0; i < kSfPrefetch - 1; ++i) ring[i] = ring[i + 1];
        ring[kSfPrefetch - 1] = fetch();
        // the stage's activation copies have landed: the scales of the terms are
        // in shared memory, and the MMAs that read this stage's TMEM scale
        // columns before are complete (the copies waited for them); the
        // weight tile may still be on its way from HBM
        if (!mbar_wait<false, true>(bfull_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
        // a reused slot: the MMAs of stage g - SLOTS have read it
        if constexpr (C::DECOUPLED) {
          if (g >= SLOTS && !mbar_wait<false, true>(sffree_bar(slot), sphase ^ 1u, abort_flag, a.err)) {
            ok = false;
            break;
          }
        }
        const uint32_t col = (uint32_t)(C::TMEM_SF0 + slot * C::SF_COLS);
        // weight row 32q + lane: K step s at column col + 4s + q
        tmem_st_x1(lane_base + col + 0u + q, wa.x);
        tmem_st_x1(lane_base + col + 4u + q, wa.y);
        tmem_st_x1(lane_base + col + 8u + q, wa.z);
        tmem_st_x1(lane_base + col + 12u + q, wa.w);
        // activation rows 32c + lane of every term, replicated in each lane quarter:
        // term j, K step s at columns col + 16 + 16j + 4s + c
        const uint8_t* sfb = gbase + stage * C::STAGE + A_STAGE_BYTES + NT * C::B_TERM;
        if constexpr (C::MERGE) {
          // the stacked rows n = j * r16 + i (term j, tile row i): K step s at
          // column col + 16 + SFB_STEP * s + n / 32 (rows past NT * r16: unused)
          constexpr int CH = C::SFB_STEP;
          uint4 r4[CH];
#pragma unroll
          for (int c = 0; c < CH; ++c)
            r4[c] = c < C::SFB_ROW_CHUNKS ? *reinterpret_cast<const uint4*>(sfb + (32 * c + lane) * 16)
                                          : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t cs = col + 16u;
          if constexpr (CH == 4) {
            tmem_st_x4(lane_base + cs + 0u, r4[0].x, r4[1].x, r4[2].x, r4[3].x);
            tmem_st_x4(lane_base + cs + 4u, r4[0].y, r4[1].y, r4[2].y, r4[3].y);
            tmem_st_x4(lane_base + cs + 8u, r4[0].z, r4[1].z, r4[2].z, r4[3].z);
            tmem_st_x4(lane_base + cs + 12u, r4[0].w, r4[1].w, r4[2].w, r4[3].w);
          } else {
            tmem_st_x8(lane_base + cs + 0u, r4[0].x, r4[1].x, r4[2].x, r4[3].x, r4[4].x, r4[5].x, r4[6].x, r4[7].x);
            tmem_st_x8(lane_base + cs + 8u, r4[0].y, r4[1].y, r4[2].y, r4[3].y, r4[4].y, r4[5].y, r4[6].y, r4[7].y);
            tmem_st_x8(lane_base + cs + 16u, r4[0].z, r4[1].z, r4[2].z, r4[3].z, r4[4].z, r4[5].z, r4[6].z, r4[7].z);
            tmem_st_x8(lane_base + cs + 24u, r4[0].w, r4[1].w, r4[2].w, r4[3].w, r4[4].w, r4[5].w, r4[6].w, r4[7].w);
          }
        } else {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          uint4 r4[BNMAX / 32];
#pragma unroll
          for (int c = 0; c < BNMAX / 32; ++c)   // (rows past the tile read other terms' scales: unused)
            r4[c] = *reinterpret_cast<const uint4*>(sfb + (j * r16 + 32 * c + lane) * 16);
          const uint32_t cj = col + 16u + 16u * j;
          if constexpr (BNMAX == 32) {
            tmem_st_x1(lane_base + cj + 0u, r4[0].x);
            tmem_st_x1(lane_base + cj + 4u, r4[0].y);
            tmem_st_x1(lane_base + cj + 8u, r4[0].z);
            tmem_st_x1(lane_base + cj + 12u, r4[0].w);
          } else if constexpr (BNMAX == 64) {
            tmem_st_x2(lane_base + cj + 0u, r4[0].x, r4[1].x);
            tmem_st_x2(lane_base + cj + 4u, r4[0].y, r4[1].y);
            tmem_st_x2(lane_base + cj + 8u, r4[0].z, r4[1].z);
            tmem_st_x2(lane_base + cj + 12u, r4[0].w, r4[1].w);
          } else {
            tmem_st_x4(lane_base + cj + 0u, r4[0].x, r4[1].x, r4[2].x, r4[3].x);
            tmem_st_x4(lane_base + cj + 4u, r4[0].y, r4[1].y, r4[2].y, r4[3].y);
            tmem_st_x4(lane_base + cj + 8u, r4[0].z, r4[1].z, r4[2].z, r4[3].z);
            tmem_st_x4(lane_base + cj + 12u, r4[0].w, r4[1].w, r4[2].w, r4[3].w);
          }
        }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(sf_bar(slot));
        ++g;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        if (++slot == SLOTS) { slot = 0; sphase ^= 1u; }
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ---------------- epilogue: warps 2..5, TMEM lane quarter = warp % 4 ----------------
    const int q = warp & 3;
    uint8_t* stg = epi_smem + q * C::EPI_WARP;
    float* wrow = reinterpret_cast<float*>(stg + C::STG);
    float* grow = wrow + BNMAX;
    const CUtensorMap* out_map = tma_out ? &maps.out : nullptr;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit; t < total; t += n_units) {
      Tile ti;
      tile_of((t - unit) / n_units, t, walk, ti);
      // the rows' scales (and routing weights), fetched while the MMAs run
      __syncwarp();
      for (int r = lane; r < ti.rows; r += 32) {
        const int row = ti.row0 + r;
        grow[r] = a.x_scale[row];
        if (EPI == EPI_SCALE) wrow[r] = a.topw[(int64_t)a.route_token[row] * a.top_k + a.route_slot[row]];
      }
      __syncwarp();
      if (!mbar_wait<false, true>(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      tc_fence_after();
      const int f0 = ti.m0 + 32 * q;
      const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * C::ACC_COLS);
      const int r16 = (ti.rows + 15) & ~15;
      for (int c0 = 0; c0 < ti.rows; c0 += 32) {
        float v[32];
        tmem_ld32(tb + (uint32_t)c0, v);
        if constexpr (C::MERGE) {
          // the other terms' columns of the same rows, added in term order
#pragma unroll 1
          for (int j = 1; j < NT; ++j) {
            float w[32];
            tmem_ld32(tb + (uint32_t)(j * r16 + c0), w);
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] += w[c];
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] *= grow[min(c0 + c, BNMAX - 1)];
        tile_epilogue<EPI, OUT_F32, false>(a, out_map, ti, c0, f0, lane, wrow, stg, v);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(C::TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// 2-D map of a byte matrix [rows, cols] (row pitch ld bytes), boxes of
// box_rows x box_cols bytes
// 3-D map of byte planes [planes, rows, cols] (row pitch ld, plane pitch
// plane_ld bytes), boxes of every plane x box_rows x box_cols bytes
bool make_plane_map(CUtensorMap* m, const void* ptr, int planes, int64_t rows, int64_t cols, int64_t ld,
                    int64_t plane_ld, int box_cols, int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)ld, (cuuint64_t)plane_ld};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, (cuuint32_t)planes};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_byte_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                   int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Fp4Key {
  const void* w;
  int64_t w_rows;
  int k;
  const void* x;
  const void* x_sf;
  int64_t x_rows;                    // rows of one term
  int terms;
  int64_t sf_ld;
  const void* out;
  int64_t out_rows, out_ld;
  int n, out_f32;
  bool operator==(const Fp4Key& o) const { return memcmp(this, &o, sizeof(Fp4Key)) == 0; }
};

bool get_fp4_maps(const Fp4Key& key, Fp4Maps& out, int& tma_out) {
  constexpr int kSlots = 16;
  static std::mutex mu;
  static Fp4Key keys[kSlots];
  static Fp4Maps maps[kSlots];
  static int outs[kSlots];
  static bool used[kSlots] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < kSlots; ++i)
    if (used[i] && keys[i] == key) {
      out = maps[i];
      tma_out = outs[i];
      return true;
    }
  Fp4Maps m;
  memset(&m, 0, sizeof(m));
  if (!make_byte_map(&m.a, key.w, key.w_rows, key.k / 2, key.k / 2, ROW_BYTES, BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  for (int i = 0; i < N_HEIGHTS; ++i) {
    if (!make_plane_map(&m.b[i], key.x, key.terms, key.x_rows, key.k / 2, key.k / 2, key.x_rows * (key.k / 2),
                        ROW_BYTES, 16 * (i + 1), CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
    if (!make_plane_map(&m.sfb[i], key.x_sf, key.terms, key.x_rows, key.k / 16, key.sf_ld, key.x_rows * key.sf_ld,
                        16, 16 * (i + 1), CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
  }
  const int to = make_out_map(&m.out, key.out, key.out_rows, key.n, key.out_ld, key.out_f32 != 0) ? 1 : 0;
  keys[next] = key;
  maps[next] = m;
  outs[next] = to;
  used[next] = true;
  next = (next + 1) % kSlots;
  out = m;
  tma_out = to;
  return true;
}

template <int EPI, bool OUT_F32, int BNMAX, int NT>
cudaError_t launch_fp4_t(const Fp4Maps& maps, const GemvArgs& a, int E, int m_tiles, int bn, int units, int to,
                         cudaStream_t s) {
  using C = Fp4Cfg<BNMAX, NT>;
  auto kernel = fp4_gemm_kernel<EPI, OUT_F32, BNMAX, NT>;
  const size_t smem = (size_t)C::STAGES * C::STAGE + C::fixed_smem(1024);
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([&](int&) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  return launch_k(kernel, units * C::CPS, kFp4Threads, smem, s, maps, a, E, m_tiles, bn, to);
}

template <int EPI, bool OUT_F32, int NT>
cudaError_t launch_fp4_bn(const Fp4Maps& maps, const GemvArgs& a, int E, int m_tiles, int bn, int units, int to,
                          cudaStream_t s) {
  if (bn <= 16) return launch_fp4_t<EPI, OUT_F32, 16, NT>(maps, a, E, m_tiles, bn, units, to, s);
  if (bn <= 32) return launch_fp4_t<EPI, OUT_F32, 32, NT>(maps, a, E, m_tiles, bn, units, to, s);
  return launch_fp4_t<EPI, OUT_F32, 64, NT>(maps, a, E, m_tiles, bn, units, to, s);
}

}  // namespace

cudaError_t launch_quant_terms(const void* x, int64_t x_ld, const int32_t* gather, const int32_t* count, int R, int K,
                               int nterms, uint8_t* q, uint8_t* sf, float* g, int64_t rows_cap, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  if (K % 64 || x_ld % 8 || rows_cap < R) return cudaErrorNotSupported;
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(R, 8), 8192);
  const int64_t ld = act_sf_ld(K);
  const bf16* xb = reinterpret_cast<const bf16*>(x);
  switch (nterms) {
    case 1: launch_k(quant_terms_kernel<1>, grid, 256, 0, s, xb, x_ld, gather, count, R, K, q, sf, g, rows_cap, ld); break;
    case 2: launch_k(quant_terms_kernel<2>, grid, 256, 0, s, xb, x_ld, gather, count, R, K, q, sf, g, rows_cap, ld); break;
    case 3: launch_k(quant_terms_kernel<3>, grid, 256, 0, s, xb, x_ld, gather, count, R, K, q, sf, g, rows_cap, ld); break;
    case 4: launch_k(quant_terms_kernel<4>, grid, 256, 0, s, xb, x_ld, gather, count, R, K, q, sf, g, rows_cap, ld); break;
    default: return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

// Rows per tile: 16 or 32 where the segments hold few rows (decode: an
// expert's rows fit one tile, and the kernels for short tiles keep more weight
// stages in flight), else 64 (with three terms stacked, 192 MMA columns);
// fewer when the product is too small to give every SM two tiles.
int fp4_tile_rows(int64_t rows_per_seg, int64_t segs, int N) {
  const int64_t m_tiles = ceil_div(N, BM);
  const int64_t units = num_sms();
  const int64_t rows = std::max<int64_t>(rows_per_seg, 1);
  int bn = rows <= 16 ? 16 : rows <= 32 ? 32 : 64;
  while (bn > 16 && ceil_div(rows, bn) * segs * m_tiles < 2 * units) bn -= 16;
  return bn;
}

cudaError_t launch_gemm_fp4(const GemvArgs& a, int epi, bool out_f32, int64_t w_rows, int E, int bn, cudaStream_t s) {
  if (a.K % 64 || a.N % 32 || bn < 16 || bn > 64 || bn % 16 || E > 1024 || !a.W_sf || !a.X_sf || !a.x_scale)
    return cudaErrorNotSupported;
  if (a.x_terms < 1 || a.x_terms > kActTermsMax || a.x_rows_cap <= 0 || a.x_sf_ld % 16 || a.x_sf_ld < a.K / 16)
    return cudaErrorNotSupported;
  if (a.K % 128) return cudaErrorNotSupported;        // weight-scale rows 8-byte aligned
  const bool of32 = out_f32 || epi == EPI_SCALE;
  const int64_t out_rows = a.offsets ? a.x_rows_cap : a.dense_rows;
  Fp4Maps maps;
  int to = 0;
  Fp4Key key;
  memset(&key, 0, sizeof(key));
  key.w = a.W; key.w_rows = w_rows; key.k = a.K; key.x = a.X; key.x_sf = a.X_sf;
  key.x_rows = a.x_rows_cap; key.terms = a.x_terms; key.sf_ld = a.x_sf_ld; key.out = a.out; key.out_rows = out_rows;
  key.out_ld = a.out_ld; key.n = a.N; key.out_f32 = of32 ? 1 : 0;
  if (!get_fp4_maps(key, maps, to)) return cudaErrorInvalidValue;
  const int m_tiles = (a.N + BM - 1) / BM;
  int units = num_sms();
  if (!a.offsets) units = (int)std::min<int64_t>(units, ceil_div(a.dense_rows, bn) * m_tiles);
  if (units <= 0) return cudaSuccess;
#define MOE_FP4(NT_)                                                                                       \
  do {                                                                                                     \
    if (epi == EPI_RELU2 && !out_f32) return launch_fp4_bn<EPI_RELU2, false, NT_>(maps, a, E, m_tiles, bn, units, to, s); \
    if (epi == EPI_SCALE) return launch_fp4_bn<EPI_SCALE, true, NT_>(maps, a, E, m_tiles, bn, units, to, s);           \
    return cudaErrorNotSupported;                                                                          \
  } while (0)
  switch (a.x_terms) {
    case 1: MOE_FP4(1);
    case 2: MOE_FP4(2);
    case 3: MOE_FP4(3);
    case 4: MOE_FP4(4);
    default: return cudaErrorNotSupported;
  }
#undef MOE_FP4
}

}  // namespace moe
