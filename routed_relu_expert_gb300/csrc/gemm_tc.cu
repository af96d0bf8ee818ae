// Tensor-core grouped GEMM for segments with many rows (prefill):
//   out[row, f] = epilogue( sum_k X[row, k] * W_seg[f, k] )
// computed as D^T = W_tile (A, 128 features x K) * X_tile^T (B, up to 256 rows)
// with tcgen05.mma (kind::f16, BF16 in, FP32 accumulate in TMEM).
//
// One persistent CTA per SM walks the tile list (segment, 128-feature tile,
// row tile).  Warp 0 streams A and B tiles with TMA (128-byte swizzle,
// K-major, 64 K-elements per stage) through a 4-stage shared-memory ring;
// one thread of warp 1 issues the MMAs; warps 2-5 read the accumulator from
// TMEM and run the epilogue, which overlaps the next tile's MMAs through two
// TMEM accumulators.  Row tiles end at segment boundaries: rows a tile loads
// beyond its segment are computed and discarded, and the MMA N is the row
// count rounded up to 16, so small tail tiles cost little.
//
// Every wait on an mbarrier gives up after a time limit: the waiter sets
// MOE_DEVERR_TIMEOUT and an abort flag that stops the other roles, the
// producer waits (bounded) for its copies in flight, the MMA thread for its
// MMAs, and the CTA frees its TMEM and returns.
//
// "One GEMM pair an expert" (page "NemotronH (Nemotron 3.5 Lightning, Bolt,
// Super VL)", section "Super VL", prefill bullet; section "Lightning",
// prefill bullet) is the prior art; here all experts' tiles form one launch.
#include "epilogue.cuh"
#include "nvfp4.cuh"

#include <cuda.h>

#include <cstring>
#include <mutex>

namespace moe {

namespace {

constexpr int BM = 128;                        // features per tile (MMA M)
constexpr int BK = 64;                         // K per stage: one 128-byte swizzle row
constexpr int BN_MAX = 256;                    // rows per tile (MMA N at most)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int B_BYTES = BN_MAX * BK * 2;       // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int N_BOX = 5;                       // B boxes of 16, 32, 64, 128, 256 rows: a tile's rows,
                                               // rounded up to 16, load as their binary decomposition
constexpr int kThreads = 192;                  // TMA, MMA, 4 epilogue warps
constexpr int kConvThreads = 128;              // NVFP4 A converters: one thread per tile row
constexpr int kThreadsFp4 = kThreads + kConvThreads;
constexpr uint32_t TMEM_COLS = 512;            // two accumulators of BN_MAX columns
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr int kMaxSegments = 1024;

struct TcMaps {
  CUtensorMap a;
  CUtensorMap b[N_BOX];
};

// ---------------------------------------------------------------------------
// PTX wrappers
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

// Bounded wait for the phase of `parity` to complete; false if this thread
// gave up or another role raised the abort flag.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      set_error(err, MOE_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
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

// Instruction descriptor, kind::f16: BF16 A and B (K-major), FP32 D, M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
struct Tile {
  int seg, m0, row0, rows;
};

__device__ __forceinline__ void decode_tile(int t, const int* prefix, int E, int m_tiles, int bn, const GemvArgs& a,
                                            Tile& ti) {
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
    base = a.offsets[lo];
    count = a.offsets[lo + 1] - base;
  }
  ti.seg = seg;
  ti.m0 = m * BM;
  ti.row0 = base + nt * bn;
  ti.rows = min(bn, count - nt * bn);
}

// Epilogue of 32 accumulator columns (rows row0+c0 .. +31) of one feature f.
// Per-row inputs are fetched before any store: the routing weight of each
// column by one lane and broadcast, the added term as 32 independent loads.
template <int EPI, bool OUT_F32>
__device__ __forceinline__ void tile_epilogue(const GemvArgs& a, const Tile& ti, int c0, int f, bool fv, int lane,
                                              float (&v)[32]) {
  const int nc = min(32, ti.rows - c0);
  if (EPI == EPI_SCALE) {
    float wl = 0.f;
    if (lane < nc) {
      const int r = ti.row0 + c0 + lane;
      wl = a.topw[(int64_t)a.route_token[r] * a.top_k + a.route_slot[r]];
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] *= __shfl_sync(0xffffffffu, wl, c);
  }
  if (!fv) return;
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
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if (c >= nc) break;
    float r = v[c];
    if (EPI == EPI_RELU2) {
      const float u = fmaxf(round_bf16(r), 0.f);
      r = u * u;
    }
    const int64_t o = (int64_t)(ti.row0 + c0 + c) * a.out_ld + f;
    if (OUT_F32 || EPI == EPI_SCALE)
      reinterpret_cast<float*>(a.out)[o] = r;
    else
      reinterpret_cast<bf16*>(a.out)[o] = __float2bfloat16_rn(r);
  }
}

// FP4A: the A operand (weights) is NVFP4 (a.W packed bytes, a.W_sf E4M3 block
// scales) and warps 6..9 turn each 128 x 64 stage into BF16 in shared memory
// (value * block scale, exact), in the 128-byte-swizzled layout TMA would have
// written; the per-tensor scale is applied by the epilogue.
template <int EPI, bool OUT_F32, bool FP4A>
__global__ void __launch_bounds__(FP4A ? kThreadsFp4 : kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, const GemvArgs a, int E, int m_tiles, int bn, int b_period) {
  constexpr int NTHR = FP4A ? kThreadsFp4 : kThreads;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto tempty_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + s); };   // FP4A: A tile converted
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* scan_tmp = reinterpret_cast<int*>(tmem_holder + 4);          // [16]
  int* prefix = scan_tmp + 16;                                         // [E+1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull_bar(i), 1);
      mbar_init(tempty_bar(i), 128);
    }
    mbar_init(drain_bar, 1);
    if (FP4A)
      for (int s = 0; s < STAGES; ++s) mbar_init(afull_bar(s), kConvThreads);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // barriers and TMEM are set up while the previous kernel finishes; its
  // results (offsets, activations) are read only after this wait
  pdl_wait();
  // row-tile prefix over segments (each segment: ceil(rows / bn) row tiles)
  int total_q;
  if (a.offsets) {
    const int per = (E + NTHR - 1) / NTHR;
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
    if (threadIdx.x == NTHR - 1) prefix[E] = wbase + x;
    // (e0 >= E for the last threads: they still write prefix[E] correctly as the block total)
  } else {
    total_q = (a.dense_rows + bn - 1) / bn;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (a.offsets) total_q = prefix[E];
  const uint32_t tmem_base = *tmem_holder;
  const int total = total_q * m_tiles;
  const int nkb = a.K / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int pend[STAGES];
      for (int s = 0; s < STAGES; ++s) pend[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile ti;
        decode_tile(t, prefix, E, m_tiles, bn, a, ti);
        const int r16 = (ti.rows + 15) & ~15;
        const uint32_t bbytes = (uint32_t)r16 * BK * 2;
        const int a_row = ti.seg * a.N + ti.m0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
          const uint32_t sa = base + stage * STAGE_BYTES;
          mbar_expect_tx(full_bar(stage), (FP4A ? 0u : (uint32_t)A_BYTES) + bbytes);
          if (!FP4A) tma_load_2d(sa, &maps.a, kb * BK, a_row, full_bar(stage));
          int off = 0;
#pragma unroll
          for (int i = N_BOX - 1; i >= 0; --i) {
            if (r16 & (16 << i)) {
              tma_load_2d(sa + A_BYTES + off * (BK * 2), &maps.b[i], (kb % b_period) * BK, ti.row0 + off,
                          full_bar(stage));
              off += 16 << i;
            }
          }
          pend[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // copies still in flight must land before the CTA leaves
        for (int s = 0; s < STAGES; ++s) {
          if (pend[s] < 0) continue;
          const uint64_t t0 = globaltimer();
          while (!mbar_try(full_bar(s), (uint32_t)pend[s]) && globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile ti;
        decode_tile(t, prefix, E, m_tiles, bn, a, ti);
        const uint32_t idesc = idesc_bf16(BM, (ti.rows + 15) & ~15);
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN_MAX);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
          if (FP4A && !mbar_wait(afull_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE_BYTES;
          const uint64_t da = smem_desc_sw128(sa), db = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma(d, da + 2u * k, db + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
          issued = true;
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && issued) {
        // MMAs still reading shared memory / writing TMEM must finish first
        tc_commit(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try(drain_bar, 0u) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (FP4A && warp >= kThreads / 32) {
    // ------- NVFP4 A converters: warps 6..9; thread = tile row, 64 values per stage -------
    const int r = threadIdx.x - kThreads;            // tile row
    const int64_t rowb = a.K / 2, rows_sf = a.K / 16;
    const uint8_t* Wq = reinterpret_cast<const uint8_t*>(a.W);
    // flat sequence of (tile, k block) items; loads run two items ahead
    struct Item { uint4 q0, q1; uint32_t sc; };
    int ft = blockIdx.x, fkb = 0;                    // fetch cursor and its tile
    Tile fti;
    if (ft < total) decode_tile(ft, prefix, E, m_tiles, bn, a, fti);
    auto fetch_next = [&](Item& it) {
      const int f = fti.m0 + r;
      if (f < a.N) {
        const int64_t row = (int64_t)fti.seg * a.N + f;
        const uint8_t* src = Wq + row * rowb + fkb * (BK / 2);
        it.q0 = ldg_stream(src);
        it.q1 = ldg_stream(src + 16);
        it.sc = __ldg(reinterpret_cast<const uint32_t*>(a.W_sf + row * rows_sf + fkb * (BK / 16)));
      } else {
        it.q0 = it.q1 = make_uint4(0, 0, 0, 0);
        it.sc = 0;
      }
      if (++fkb == nkb) {
        fkb = 0;
        ft += gridDim.x;
        if (ft < total) decode_tile(ft, prefix, E, m_tiles, bn, a, fti);
      }
    };
    Item cur, nxt;
    cur.q0 = cur.q1 = nxt.q0 = nxt.q1 = make_uint4(0, 0, 0, 0);
    cur.sc = nxt.sc = 0;
    if (ft < total) fetch_next(cur);
    if (ft < total) fetch_next(nxt);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb) {
        Item nn = cur;
        if (ft < total) fetch_next(nn);
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
        const uint32_t s0 = e4m3x2_to_f16x2(cur.sc & 0xFFFFu), s1 = e4m3x2_to_f16x2(cur.sc >> 16);
        const uint32_t sc[4] = {__byte_perm(s0, 0, 0x1010), __byte_perm(s0, 0, 0x3232),
                                __byte_perm(s1, 0, 0x1010), __byte_perm(s1, 0, 0x3232)};
        const uint32_t w[8] = {cur.q0.x, cur.q0.y, cur.q0.z, cur.q0.w, cur.q1.x, cur.q1.y, cur.q1.z, cur.q1.w};
        uint8_t* dst = gbase + stage * STAGE_BYTES + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {            // 16-byte chunk c = values 8c .. 8c+7
          uint32_t p[4];
          e2m1x8_to_f16x2(w[c], p);
          uint4 o;
          o.x = f16x2_to_bf16x2(hmul2_f16(p[0], sc[c >> 1]));
          o.y = f16x2_to_bf16x2(hmul2_f16(p[1], sc[c >> 1]));
          o.z = f16x2_to_bf16x2(hmul2_f16(p[2], sc[c >> 1]));
          o.w = f16x2_to_bf16x2(hmul2_f16(p[3], sc[c >> 1]));
          *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) = o;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(afull_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        cur = nxt;
        nxt = nn;
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ---------------- epilogue: warps 2..5, TMEM lane quarter = warp % 4 ----------------
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      Tile ti;
      decode_tile(t, prefix, E, m_tiles, bn, a, ti);
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      tc_fence_after();
      const int f = ti.m0 + 32 * q + lane;
      const bool fv = f < a.N;
      const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN_MAX);
      for (int c0 = 0; c0 < ti.rows; c0 += 32) {
        float v[32];
        tmem_ld32(tb + (uint32_t)c0, v);
        tile_epilogue<EPI, OUT_F32>(a, ti, c0, f, fv, lane, v);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld_elems, int box_rows) {
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

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

size_t smem_bytes(int E) {
  return 1024 + (size_t)STAGES * STAGE_BYTES + (3 * STAGES + 5) * 8 + 16 + (16 + E + 1) * sizeof(int) + 64;
}

template <int EPI, bool OUT_F32, bool FP4A>
cudaError_t launch_t(const TcMaps& maps, const GemvArgs& a, int E, int m_tiles, int bn, int b_period, int grid,
                     cudaStream_t s) {
  const size_t smem = smem_bytes(kMaxSegments);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<EPI, OUT_F32, FP4A>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(tc_gemm_kernel<EPI, OUT_F32, FP4A>, grid, FP4A ? kThreadsFp4 : kThreads, smem, s, maps, a, E,
                  m_tiles, bn, b_period);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemvArgs& a, int epi, bool out_f32, int64_t w_rows, int64_t x_rows, int E, int bn,
                           cudaStream_t s, int x_cols) {
  if (a.K % BK != 0 || bn < 16 || bn > BN_MAX || (bn & (bn - 1)) || E > kMaxSegments) return cudaErrorNotSupported;
  if (x_cols <= 0) x_cols = a.K;
  if (x_cols % BK != 0 || a.K % x_cols != 0) return cudaErrorNotSupported;
  const bool fp4 = a.W_sf != nullptr;       // NVFP4 weights: converted in the kernel
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (!fp4 && !make_map(&maps.a, a.W, w_rows, a.K, a.K, BM)) return cudaErrorInvalidValue;
  for (int i = 0; i < N_BOX; ++i)
    if (!make_map(&maps.b[i], a.X, x_rows, x_cols, a.x_ld, 16 << i)) return cudaErrorInvalidValue;
  const int m_tiles = (a.N + BM - 1) / BM;
  const int b_period = x_cols / BK;
  int grid = num_sms();
  if (!a.offsets) grid = (int)std::min<int64_t>(grid, ceil_div(a.dense_rows, bn) * m_tiles);
  if (grid <= 0) return cudaSuccess;
  if (fp4) {
    switch (epi) {
      case EPI_RELU2: return launch_t<EPI_RELU2, false, true>(maps, a, E, m_tiles, bn, b_period, grid, s);
      case EPI_SCALE: return launch_t<EPI_SCALE, true, true>(maps, a, E, m_tiles, bn, b_period, grid, s);
      default: return cudaErrorNotSupported;
    }
  }
  switch (epi) {
    case EPI_RELU2: return launch_t<EPI_RELU2, false, false>(maps, a, E, m_tiles, bn, b_period, grid, s);
    case EPI_SCALE: return launch_t<EPI_SCALE, true, false>(maps, a, E, m_tiles, bn, b_period, grid, s);
    case EPI_STORE:
      return out_f32 ? launch_t<EPI_STORE, true, false>(maps, a, E, m_tiles, bn, b_period, grid, s)
                     : launch_t<EPI_STORE, false, false>(maps, a, E, m_tiles, bn, b_period, grid, s);
    default:
      return out_f32 ? launch_t<EPI_ADD, true, false>(maps, a, E, m_tiles, bn, b_period, grid, s)
                     : launch_t<EPI_ADD, false, false>(maps, a, E, m_tiles, bn, b_period, grid, s);
  }
}

}  // namespace moe
