// Tensor-core grouped GEMM for segments with many rows (prefill):
//   out[row, f] = epilogue( sum_k X[row, k] * W_seg[f, k] )
// computed as D^T = W_tile (A, features x K) * X_tile^T (B, up to 256 rows)
// with tcgen05.mma (kind::f16, BF16 in, FP32 accumulate in TMEM).
//
// Persistent kernel: one CTA per SM, or one CTA pair per two SMs, walks the
// tile list (segment, feature tile, row tile).  Warps 0 and 6 stream the A and
// the B tiles with TMA (128-byte swizzle, K-major, 64 K-elements per stage)
// through a shared-memory ring: one TMA box per operand and stage, each issued
// by its own warp, since one issuing thread sustains only about one box per
// 300-400 cycles.  One thread of warp 1 issues the MMAs; warps 2-5 read the
// accumulator from TMEM and run the epilogue, which overlaps the next tile's
// MMAs through two TMEM accumulators.  Row tiles end at segment boundaries:
// rows a tile loads beyond its segment are computed and discarded, and the MMA
// N is the row count rounded up to 16, so small tail tiles cost little.
//
// CG = 2 (a cluster of two CTAs on two SMs, tcgen05 cta_group::2): the tile is
// 256 features x N rows.  Each CTA stages its own 128 features of A and half
// of the N rows of B; the even CTA issues M = 256 MMAs that read both CTAs'
// shared memory and write 128 TMEM lanes in each.  Per SM this halves the B
// bytes staged per MMA, so a stage carries 32 KB instead of 48 KB for the same
// tensor work: the L2-to-SM copy rate (about 60-68 bytes per cycle per SM),
// not the tensor pipe, bounds the single-CTA form.  The even CTA's "full" barrier counts both CTAs' TMA
// bytes; MMA completion is signalled to both CTAs' "empty" and "accumulator
// full" barriers by a multicast commit; the odd CTA's epilogue threads arrive
// on the even CTA's "accumulator empty" barrier remotely.  NVFP4 weights run
// on single CTAs (see pick_cg).
//
// Every wait on an mbarrier gives up after a time limit: the waiter sets
// MOE_DEVERR_TIMEOUT and an abort flag that stops the other roles, the
// producer waits (bounded) for its copies in flight, the MMA thread for its
// MMAs, and the CTA frees its TMEM and returns.
//
// "One GEMM pair an expert" (page "NemotronH (Nemotron 3.5 Lightning, Bolt,
// Super VL)", section "Super VL", prefill bullet; section "Lightning",
// prefill bullet) is the prior art; here all experts' tiles form one launch.
#include "tc_common.cuh"

#include <cstring>
#include <mutex>

namespace moe {

namespace {

using namespace tc;

constexpr int BN_MAX = 256;                    // rows per tile (MMA N at most)
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int N_BMAP = 16;                     // B boxes of 1..16 x (16 / CG) rows: every tile's B
                                               // half loads as one box
constexpr int kThreads = 224;                  // A TMA, MMA, 4 epilogue warps, B TMA
constexpr int kBWarp = 6;
constexpr int kConvThreads = 256;              // NVFP4 A converters: two threads per tile row
constexpr int kConvChunks = 8 * BM / kConvThreads;   // 16-byte output chunks (8 values) per thread
constexpr int kThreadsFp4 = kThreads + kConvThreads;
constexpr uint32_t TMEM_COLS = 512;            // two accumulators of BN_MAX columns
constexpr int kMaxSegments = 1024;

// ring geometry per CTA group size (CG = CTAs that share one MMA); FP4A: a
// second ring of raw NVFP4 weight bytes feeds the converters
template <int CG, bool FP4A = false>
struct Ring {
  static constexpr int TILE_M = BM * CG;                  // features per tile
  static constexpr int B_ROWS = BN_MAX / CG;              // B rows one CTA stages
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB (CG 1), 32 KB (CG 2)
  static constexpr int STAGES = FP4A ? (CG == 2 ? 5 : 3) : (CG == 2 ? 6 : 4);
  static constexpr int BOX0 = 16 / CG;                    // B box height step (rows)
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int RAW_STAGES = FP4A ? 8 : 0;         // 128 rows x 32 packed bytes each
  static constexpr int RAW_BYTES = RAW_STAGES * BM * (BK / 2);
};

// epilogue staging after the ring: per epilogue warp one 32 x 32 output chunk
// (FP32 at most) and the routing weights of one tile's rows
constexpr int STG_BYTES = 32 * 32 * 4;
constexpr int WROW_BYTES = BN_MAX * 4;
constexpr int EPI_SMEM = 4 * (STG_BYTES + WROW_BYTES);

struct TcMaps {
  CUtensorMap a;
  CUtensorMap b[N_BMAP];                         // b[i]: boxes of (i + 1) * BOX0 rows
  CUtensorMap out;                               // output, boxes of 32 rows x 32 features
};

// FP4A: the A operand (weights) is NVFP4 (a.W packed bytes, a.W_sf E4M3 block
// scales) and the converter warps turn each 128 x 64 stage into BF16 (FP4A 1)
// or FP16 (FP4A 2: the B rows are FP16 too, and a BF16-activation output is
// stored as FP16 copies of its BF16 values) in shared memory (value * block
// scale, exact in either), in the 128-byte-swizzled layout TMA would have
// written; the per-tensor scale is applied by the epilogue.
template <int EPI, bool OUT_F32, int FP4A, int CG>
__global__ void __launch_bounds__(FP4A ? kThreadsFp4 : kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, const GemvArgs a, int E, int m_tiles, int bn, int b_period,
                   int tma_out, int ksplit) {
  static_assert(!(FP4A && CG == 2), "NVFP4 weights run on single CTAs");
  using G = Ring<CG, (FP4A != 0)>;
  constexpr int NTHR = FP4A ? kThreadsFp4 : kThreads;
  constexpr int STAGES = G::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint8_t* epi_smem = gbase + G::RING_BYTES;                        // 4 x (staging, row weights)
  uint8_t* raw_smem = epi_smem + EPI_SMEM;                            // FP4A: packed weight ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw_smem + G::RAW_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + s); };   // FP4A: this CTA's A converted
  constexpr int RS = G::RAW_STAGES;
  auto rfull_bar = [&](int s) { return bar0 + 8u * (4 * STAGES + 5 + s); };        // FP4A: raw bytes landed
  auto rempty_bar = [&](int s) { return bar0 + 8u * (4 * STAGES + 5 + RS + s); };  // FP4A: raw slot read
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 4 * STAGES + 5 + 2 * RS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* scan_tmp = reinterpret_cast<int*>(tmem_holder + 4);          // [16]
  int* prefix = scan_tmp + 16;                                         // [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CG 2: rank 0 of the pair issues the MMAs and owns the barriers both CTAs'
  // copies and drains arrive on; both walk the same tile sequence
  const uint32_t rank = CG == 2 ? cluster_rank() : 0u;
  const int unit = CG == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = CG == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  auto at_leader = [&](uint32_t bar) { return CG == 2 ? map_to_rank0(bar) : bar; };
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), FP4A ? 1 : 2);      // the A and B producers of CTA 0
      mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 128 * CG);
    }
    mbar_init(drain_bar, 1);
    if (FP4A) {
      for (int s = 0; s < STAGES; ++s) mbar_init(afull_bar(s), kConvThreads);
      for (int s = 0; s < RS; ++s) {
        mbar_init(rfull_bar(s), 1);
        mbar_init(rempty_bar(s), kConvThreads);
      }
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if (CG == 2) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                   "r"(TMEM_COLS)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }

  // barriers and TMEM are set up while the previous kernel finishes; its
  // results (offsets, activations) are read only after this wait
  pdl_wait();
  // row-tile prefix over segments (each segment: ceil(rows / bn) row tiles)
  if (a.offsets) row_tile_prefix(a, E, bn, NTHR, scan_tmp, prefix);
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();      // the peer's barriers exist before any remote arrive or copy
  tc_fence_after();
  const int total_q = a.offsets ? prefix[E] : (a.dense_rows + bn - 1) / bn;
  const uint32_t tmem_base = *tmem_holder;
  const int per_part = total_q * m_tiles;
  const int total = per_part * ksplit;
  const int nkb = a.K / BK;

  if (FP4A && warp == 0) {
    if (lane == 0) {
      // ------- FP4A: packed weight bytes of this CTA's 128 rows, one box per k-block -------
      int rs = 0;
      uint32_t rphase = 0;
      bool ok = true;
      int pend[RS > 0 ? RS : 1];
      for (int s = 0; s < RS; ++s) pend[s] = -1;
      for (int t = unit; t < total && ok; t += n_units) {
        Tile ti;
        decode_tile(t, prefix, E, m_tiles, G::TILE_M, bn, a, per_part, ksplit, nkb, ti);
        const int row = ti.seg * a.N + ti.m0 + BM * (int)rank;
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait(rempty_bar(rs), rphase ^ 1u, abort_flag, a.err)) { ok = false; break; }
          mbar_expect_tx(rfull_bar(rs), BM * (BK / 2));
          tma_load_2d(smem_u32(raw_smem) + rs * (BM * (BK / 2)), &maps.a, kb * (BK / 2), row, rfull_bar(rs));
          pend[rs] = (int)rphase;
          if (++rs == RS) { rs = 0; rphase ^= 1u; }
        }
      }
      if (!ok) {
        for (int s = 0; s < RS; ++s) {
          if (pend[s] < 0) continue;
          const uint64_t t0 = globaltimer();
          while (!mbar_try(rfull_bar(s), (uint32_t)pend[s]) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 0 || warp == kBWarp) {
    const bool is_a = warp == 0;
    if (lane == 0) {
      // ------- TMA producers: warp 0 the A (weight) tile, warp 6 the B (row) tile;
      // each CTA loads its own operand halves -------
      int pend[STAGES];
      for (int s = 0; s < STAGES; ++s) pend[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = unit; t < total && ok; t += n_units) {
        Tile ti;
        decode_tile(t, prefix, E, m_tiles, G::TILE_M, bn, a, per_part, ksplit, nkb, ti);
        const int r16 = (ti.rows + 15) & ~15;
        const int hb = r16 / CG;                             // B rows this CTA loads
        const CUtensorMap* map = is_a ? &maps.a : &maps.b[hb / G::BOX0 - 1];
        const uint32_t tx = is_a ? (uint32_t)CG * A_BYTES : (uint32_t)r16 * BK * 2;
        const int row = is_a ? ti.seg * a.N + ti.m0 + BM * (int)rank : ti.row0 + hb * (int)rank;
        const uint32_t dst0 = base + (is_a ? 0u : (uint32_t)A_BYTES);
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
          if (rank == 0) mbar_expect_tx(full_bar(stage), tx);
          const int col = is_a ? kb * BK : (kb % b_period) * BK;
          const uint32_t dst = dst0 + stage * G::STAGE_BYTES;
          if (CG == 2) tma_load_2d_pair(dst, map, col, row, at_leader(full_bar(stage)));
          else tma_load_2d(dst, map, col, row, full_bar(stage));
          pend[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && rank == 0) {
        // copies still in flight (both CTAs' count on these barriers) must land
        // before the CTA leaves
        for (int s = 0; s < STAGES; ++s) {
          if (pend[s] < 0) continue;
          const uint64_t t0 = globaltimer();
          while (!mbar_try(full_bar(s), (uint32_t)pend[s]) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int t = unit; t < total && ok; t += n_units) {
        Tile ti;
        decode_tile(t, prefix, E, m_tiles, G::TILE_M, bn, a, per_part, ksplit, nkb, ti);
        const uint32_t idesc = idesc_f16kind(G::TILE_M, (ti.rows + 15) & ~15, FP4A == 2);
        if (!mbar_wait<CG == 2>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN_MAX);
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
          if (FP4A && !mbar_wait(afull_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + stage * G::STAGE_BYTES;
          const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma<CG>(d, da + 2u * k, db + 2u * k, idesc, (kb != ti.kb0 || k != 0) ? 1u : 0u);
          issued = true;
          tc_commit<CG>(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit<CG>(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && issued) {
        // MMAs still reading shared memory / writing TMEM must finish first
        tc_commit<CG>(drain_bar, 1);
        const uint64_t t0 = globaltimer();
        while (!mbar_try(drain_bar, 0u) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (FP4A && warp >= kThreads / 32) {
    // ------- NVFP4 A converters: warps 7..14; two threads per tile row, 32 values each -------
    // packed bytes come from the raw ring (TMA, warp 0); the E4M3 block scales
    // (4 bytes per row and stage) are loaded here, kSP stages ahead
    constexpr int kSP = 6;
    const int ct = threadIdx.x - kThreads;
    const int r = ct % BM;                           // tile row
    const int hf = ct / BM;                          // half of the row's 64 values
    const int64_t rows_sf = a.K / 16;
    int ft = unit, fkb = 0;                          // scale fetch cursor and its tile
    Tile fti;
    if (ft < total) decode_tile(ft, prefix, E, m_tiles, G::TILE_M, bn, a, per_part, ksplit, nkb, fti);
    auto fetch_scale = [&]() -> uint32_t {
      uint32_t v = 0;
      if (ft >= total) return v;
      const int f = fti.m0 + BM * (int)rank + r;
      if (f < a.N) {
        const int64_t row = (int64_t)fti.seg * a.N + f;
        v = __ldg(reinterpret_cast<const uint32_t*>(a.W_sf + row * rows_sf + fkb * (BK / 16)));
      }
      if (++fkb == nkb) {
        fkb = 0;
        ft += n_units;
        if (ft < total) decode_tile(ft, prefix, E, m_tiles, G::TILE_M, bn, a, per_part, ksplit, nkb, fti);
      }
      return v;
    };
    uint32_t scq[kSP];
#pragma unroll
    for (int i = 0; i < kSP; ++i) scq[i] = fetch_scale();
    int stage = 0, rs = 0;
    uint32_t phase = 0, rphase = 0;
    bool ok = true;
    for (int t = unit; t < total && ok; t += n_units) {        // (NVFP4 products are never split in K)
      for (int kb = 0; kb < nkb; ++kb) {
        const uint32_t sc_word = scq[0];
#pragma unroll
        for (int i = 0; i < kSP - 1; ++i) scq[i] = scq[i + 1];
        scq[kSP - 1] = fetch_scale();
        if (!mbar_wait(rfull_bar(rs), rphase, abort_flag, a.err)) { ok = false; break; }
        const uint4 q = reinterpret_cast<const uint4*>(raw_smem + rs * (BM * (BK / 2)) + r * (BK / 2))[hf];
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
        // this half's two block scales as BF16 (FP16) pairs, exact, one per 16 values
        const uint32_t s16 = e4m3x2_to_f16x2((sc_word >> (16 * hf)) & 0xFFFFu);
        const uint32_t s2 = FP4A == 2 ? s16 : f16x2_to_bf16x2(s16);
        const uint32_t sc[2] = {__byte_perm(s2, 0, 0x1010), __byte_perm(s2, 0, 0x3232)};
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint8_t* dst = gbase + stage * G::STAGE_BYTES + r * 128;
#pragma unroll
        for (int c = 0; c < kConvChunks; ++c) {  // 16-byte chunk cc = values 8cc .. 8cc+7
          const int cc = hf * kConvChunks + c;
          uint32_t p[4];
          uint4 o;                               // value x scale: at most 6 significant bits, exact
          if (FP4A == 2) {
            e2m1x8_to_f16x2(w[c], p);
            o.x = hmul2_f16(p[0], sc[c >> 1]);
            o.y = hmul2_f16(p[1], sc[c >> 1]);
            o.z = hmul2_f16(p[2], sc[c >> 1]);
            o.w = hmul2_f16(p[3], sc[c >> 1]);
          } else {
            e2m1x8_to_bf16x2(w[c], p);
            o.x = hmul2_bf16(p[0], sc[c >> 1]);
            o.y = hmul2_bf16(p[1], sc[c >> 1]);
            o.z = hmul2_bf16(p[2], sc[c >> 1]);
            o.w = hmul2_bf16(p[3], sc[c >> 1]);
          }
          *reinterpret_cast<uint4*>(dst + ((cc ^ (r & 7)) << 4)) = o;
        }
        // order this thread's shared-memory accesses (the raw bytes read, the
        // converted row written) before the async-proxy accesses that follow the
        // arrives: the MMA reading the row and the next TMA copy into the raw
        // slot (releasing the slot before this fence let that copy overwrite
        // bytes still being read)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(afull_bar(stage));
        mbar_arrive(rempty_bar(rs));
        if (++rs == RS) { rs = 0; rphase ^= 1u; }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ---------------- epilogue: warps 2..5, TMEM lane quarter = warp % 4 ----------------
    const int q = warp & 3;
    uint8_t* stg = epi_smem + q * (STG_BYTES + WROW_BYTES);
    float* wrow = reinterpret_cast<float*>(stg + STG_BYTES);
    const CUtensorMap* out_map = tma_out ? &maps.out : nullptr;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit; t < total; t += n_units) {
      Tile ti;
      decode_tile(t, prefix, E, m_tiles, G::TILE_M, bn, a, per_part, ksplit, nkb, ti);
      if (EPI == EPI_SCALE) {
        // routing weights of the tile's rows, fetched while the MMAs run
        __syncwarp();
        for (int r = lane; r < ti.rows; r += 32) {
          const int row = ti.row0 + r;
          wrow[r] = a.topw[(int64_t)a.route_token[row] * a.top_k + a.route_slot[row]];
        }
        __syncwarp();
      }
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      tc_fence_after();
      const int f0 = ti.m0 + BM * (int)rank + 32 * q;
      const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN_MAX);
      for (int c0 = 0; c0 < ti.rows; c0 += 32) {
        float v[32];
        tmem_ld32(tb + (uint32_t)c0, v);
        tile_epilogue<EPI, OUT_F32, FP4A == 2>(a, out_map, ti, c0, f0, lane, wrow, stg, v);
      }
      // TMEM reads are complete (tcgen05.wait::ld); the stores need no ordering
      // with the next MMAs, so the peer's arrive is relaxed
      tc_fence_before();
      if (rank == 0) mbar_arrive(tempty_bar(acc));
      else mbar_arrive_cluster_relaxed(at_leader(tempty_bar(acc)));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) bulk_wait_all();        // this warp's output stores are complete
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();      // no CTA leaves while its peer may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    if (CG == 2)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                   : "memory");
  }
  if (CG == 2) cluster_sync();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Tensor maps of one product (A: weights, 128-row boxes; B: rows, boxes of
// 1..16 x 16/cg rows), encoded once per distinct set of pointers and extents.
struct MapKey {
  const void* w;
  int64_t w_rows;
  int k;
  const void* x;
  int64_t x_rows;
  int x_cols;
  int64_t x_ld;
  int cg;
  const void* out;                 // output [x_rows, out_ld], n features per row
  int64_t out_ld;
  int n;
  int out_f32;
  int fp4;                         // w: packed NVFP4 bytes [w_rows, k / 2]
  int64_t out_rows;                // rows of the output (K parts stack their slabs)
  bool operator==(const MapKey& o) const {
    return w == o.w && w_rows == o.w_rows && k == o.k && x == o.x && x_rows == o.x_rows && x_cols == o.x_cols &&
           x_ld == o.x_ld && cg == o.cg && out == o.out && out_ld == o.out_ld && n == o.n && out_f32 == o.out_f32 &&
           fp4 == o.fp4 && out_rows == o.out_rows;
  }
};

bool get_maps(const MapKey& key, TcMaps& out, int& tma_out) {
  constexpr int kSlots = 16;
  static std::mutex mu;
  static MapKey keys[kSlots];
  static TcMaps maps[kSlots];
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
  TcMaps m;
  memset(&m, 0, sizeof(m));
  if (key.fp4 ? !make_packed_map(&m.a, key.w, key.w_rows, key.k) : !make_map(&m.a, key.w, key.w_rows, key.k, key.k, BM))
    return false;
  for (int i = 0; i < N_BMAP; ++i)
    if (!make_map(&m.b[i], key.x, key.x_rows, key.x_cols, key.x_ld, (i + 1) * (16 / key.cg))) return false;
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

template <int CG, bool FP4A>
size_t smem_bytes(int E) {
  using G = Ring<CG, FP4A>;
  return 1024 + (size_t)G::RING_BYTES + EPI_SMEM + G::RAW_BYTES + (4 * G::STAGES + 5 + 2 * G::RAW_STAGES) * 8 + 16 +
         (16 + E + 1) * sizeof(int) + 64;
}

// Largest number of CTA pairs (clusters of 2) resident at once; 0 if unknown.
template <class K>
int max_pairs(K kernel, size_t smem, int threads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int EPI, bool OUT_F32, int FP4A, int CG>
cudaError_t launch_t(const TcMaps& maps, const GemvArgs& a, int E, int m_tiles, int bn, int b_period, int units,
                     int tma_out, int ksplit, cudaStream_t s) {
  auto kernel = tc_gemm_kernel<EPI, OUT_F32, FP4A, CG>;
  const size_t smem = smem_bytes<CG, (FP4A != 0)>(kMaxSegments);
  const int threads = FP4A ? kThreadsFp4 : kThreads;
  // shared-memory limit set once per device, and the CTAs (CG 1) or CTA pairs
  // (CG 2) resident at once on it
  static PerDeviceOnce cap;
  int cap_units = 0;
  const cudaError_t ce = cap.run(
      [&](int& v) -> cudaError_t {
        const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (CG == 2) {
          const int p = max_pairs(kernel, smem, threads);
          v = p > 0 ? p : num_sms() / 2;
        } else {
          v = num_sms();
        }
        return cudaSuccess;
      },
      &cap_units);
  if (ce != cudaSuccess) return ce;
  units = std::max(1, std::min(units, cap_units));
  if (CG == 1) return launch_k(kernel, units, threads, smem, s, maps, a, E, m_tiles, bn, b_period, tma_out, ksplit);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * units);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, kernel, maps, a, E, m_tiles, bn, b_period, tma_out, ksplit);
}

// fp4: 0 BF16 weights, 1 NVFP4 weights with BF16 operands, 2 NVFP4 weights
// with FP16 operands (FP16 B rows; a ReLU^2 output stored as FP16)
template <int CG>
cudaError_t launch_cg(const TcMaps& maps, const GemvArgs& a, int epi, bool out_f32, int fp4, int E, int m_tiles,
                      int bn, int b_period, int units, int to, int ks, cudaStream_t s) {
  if (fp4) {
    if constexpr (CG == 1) {
      if (fp4 == 2) {
        switch (epi) {
          case EPI_RELU2: return launch_t<EPI_RELU2, false, 2, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
          case EPI_SCALE: return launch_t<EPI_SCALE, true, 2, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
          default: return cudaErrorNotSupported;
        }
      }
      switch (epi) {
        case EPI_RELU2: return launch_t<EPI_RELU2, false, 1, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
        case EPI_SCALE: return launch_t<EPI_SCALE, true, 1, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
        default: return cudaErrorNotSupported;
      }
    }
    return cudaErrorNotSupported;
  }
  switch (epi) {
    case EPI_RELU2: return launch_t<EPI_RELU2, false, 0, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
    case EPI_SCALE: return launch_t<EPI_SCALE, true, 0, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
    case EPI_STORE:
      return out_f32 ? launch_t<EPI_STORE, true, 0, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s)
                     : launch_t<EPI_STORE, false, 0, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
    default:
      return out_f32 ? launch_t<EPI_ADD, true, 0, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s)
                     : launch_t<EPI_ADD, false, 0, CG>(maps, a, E, m_tiles, bn, b_period, units, to, ks, s);
  }
}

// CTA pairs for BF16 products with more than one 128-feature tile per
// segment.  NVFP4 weights stay on single CTAs: a pair's MMA would wait for the
// peer CTA's converted rows, and that cross-CTA hand-off cost more than the
// halved B traffic saves.
inline int pick_cg(int N, bool fp4) { return !fp4 && N > BM ? 2 : 1; }

}  // namespace

// Rows per tile: the largest power of two that still gives every unit two
// tiles (the slack balances ragged segments).  Dense products (one segment,
// uniform tiles) take instead the height with the least estimated time when it
// is clearly (15 %) better: waves x per-tile time, a tile's time per 64-deep
// k-block being the larger of its MMA cycles (128 x bn x 64 x 2 FLOP per SM at
// ~6,100 FLOP/cycle) and its shared-memory fill cycles ((128 + bn / cg) x
// 128 B per SM at ~65 B/cycle from L2, the TMA rate measured on this part).
// Short tiles re-read the weight tile once per row tile; tall ones leave SMs
// idle when there are few feature tiles (a 1024-feature projection of 4096
// rows: 64-row tiles read its weights 64 times, 256-row tiles 16 times).
int tc_tile_rows(int64_t rows_per_seg, int64_t segs, int N) {
  const int cg = pick_cg(N, false);
  const int64_t m_tiles = ceil_div(N, (int64_t)BM * cg);
  const int64_t units = num_sms() / cg;
  const int64_t rows = std::max<int64_t>(rows_per_seg, 1);
  int bn = BN_MAX;
  while (bn > 16 && ceil_div(rows, bn) * segs * m_tiles < 2 * units) bn >>= 1;
  if (segs > 1) return bn;
  auto est = [&](int b) {
    const double mma = 128.0 * b * 128.0 / 6100.0;
    const double fill = (128.0 + (double)b / cg) * 128.0 / 65.0;
    return (double)ceil_div(ceil_div(rows, b) * m_tiles, units) * std::max(mma, fill);
  };
  int best = bn;
  for (int b = BN_MAX; b >= 16; b >>= 1)
    if (est(b) < est(best)) best = b;
  return est(best) < 0.85 * est(bn) ? best : bn;
}

cudaError_t launch_gemm_tc(const GemvArgs& a, int epi, bool out_f32, int64_t w_rows, int64_t x_rows, int E, int bn,
                           cudaStream_t s, int x_cols, int ksplit) {
  if (a.K % BK != 0 || a.N % 32 != 0 || bn < 16 || bn > BN_MAX || (bn & (bn - 1)) || E > kMaxSegments)
    return cudaErrorNotSupported;
  // K parts: dense FP32 stores only, at least one k-block each
  if (ksplit < 1 || ksplit > a.K / BK || (ksplit > 1 && (a.offsets || epi != EPI_STORE || !out_f32 || a.W_sf)))
    return cudaErrorNotSupported;
  if (x_cols <= 0) x_cols = a.K;
  if (x_cols % BK != 0 || a.K % x_cols != 0) return cudaErrorNotSupported;
  const bool fp4 = a.W_sf != nullptr;       // NVFP4 weights: converted in the kernel
  // FP16 operands: NVFP4 products only, FP16 rows in and, for ReLU^2, out
  // (the tensor maps move 2-byte elements either way)
  if (a.x_f16 || a.out_f16) {
    const bool ok = fp4 && a.x_f16 && (epi == EPI_RELU2 ? a.out_f16 : epi == EPI_SCALE && !a.out_f16);
    if (!ok) return cudaErrorNotSupported;
  }
  const int cg = pick_cg(a.N, fp4);
  TcMaps maps;
  int to = 0;
  const bool of32 = out_f32 || epi == EPI_SCALE;
  if (!get_maps(MapKey{a.W, w_rows, a.K, a.X, x_rows, x_cols, a.x_ld, cg, a.out, a.out_ld, a.N, of32 ? 1 : 0,
                       fp4 ? 1 : 0, x_rows * ksplit},
                maps, to))
    return cudaErrorInvalidValue;
  const int m_tiles = (a.N + BM * cg - 1) / (BM * cg);
  const int b_period = x_cols / BK;
  int units = num_sms() / cg;
  if (!a.offsets) units = (int)std::min<int64_t>(units, ceil_div(a.dense_rows, bn) * m_tiles * ksplit);
  if (units <= 0) return cudaSuccess;
  const int fmt = fp4 ? (a.x_f16 ? 2 : 1) : 0;
  if (cg == 2) return launch_cg<2>(maps, a, epi, out_f32, fmt, E, m_tiles, bn, b_period, units, to, ksplit, s);
  return launch_cg<1>(maps, a, epi, out_f32, fmt, E, m_tiles, bn, b_period, units, to, ksplit, s);
}

}  // namespace moe
