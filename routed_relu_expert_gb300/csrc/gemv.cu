// Weight-streaming grouped GEMV for small row counts (decode).
//
// Every active expert's matrix (or one dense matrix) is read from HBM exactly
// once per call for all of that expert's rows: a CTA owns 16 output features
// of one segment, its 8 warps split the reduction dimension into 32-wide
// chunks, and the partial sums are added in a fixed warp order through shared
// memory (deterministic, no atomics).  Weight rows are fetched with 128-bit
// streaming loads; each thread's 16 bytes of row g and row g+8 feed two
// m16n8k16 MMAs whose k positions are a consistent permutation of the chunk
// (the same permutation is applied to the activation operand), so no shuffle
// or shared-memory staging is needed between the load and the MMA.
//
// The expert bank of page "NemotronH (Nemotron 3.5 Lightning, Bolt, Super
// VL)", section "How the engine runs it" (a group's CTA decodes an expert's
// tiles once for all of its rows) is the prior art; here the grouping comes
// from the dispatch offsets and the split is over features and K.
#include "epilogue.cuh"
#include "nvfp4.cuh"

#include <cuda_fp16.h>

#include <algorithm>

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct Seg {
  int id, row0, nrows;
};

// segment of this CTA: the expert id first (one level of dependent loads, so a
// caller can start its weight stream), then the rows
__device__ __forceinline__ bool resolve_id(const GemvArgs& a, Seg& s) {
  if (a.offsets) {
    const int j = blockIdx.y;
    // both loads go out together (active[] has a slot for every launched j)
    const int n_active = a.hdr->n_active;
    const int id = a.active[j];
    if (j >= n_active) return false;
    s.id = id;
  } else {
    s.id = 0;
  }
  return true;
}

__device__ __forceinline__ bool resolve_rows(const GemvArgs& a, int rows_per_cta, Seg& s) {
  if (a.offsets) {
    s.row0 = a.offsets[s.id];
    s.nrows = a.offsets[s.id + 1] - s.row0;
  } else {
    s.row0 = 0;
    s.nrows = a.dense_rows;
  }
  const int rb = blockIdx.z * rows_per_cta;
  if (rb >= s.nrows) return false;
  s.row0 += rb;
  s.nrows = min(s.nrows - rb, rows_per_cta);
  return true;
}

__device__ __forceinline__ bool resolve_segment(const GemvArgs& a, int rows_per_cta, Seg& s) {
  return resolve_id(a, s) && resolve_rows(a, rows_per_cta, s);
}

// ---------------------------------------------------------------------------
// BF16 weights, BF16 activations.  A CTA owns FPC features (16 or 32): its 8
// warps form FPC / 16 groups, a group owns 16 features and its warps split K
// in 32-wide chunks (rows short enough to leave a 16-feature CTA little work
// take 32 features, halving the CTA count and its fixed costs).  A CTA
// handles its segment's rows in passes of 16 (two 8-row MMA column blocks); a
// second pass finds the CTA's weight tile still in L2, so HBM streams each
// weight once while registers stay low.
// ---------------------------------------------------------------------------
template <int EPI, bool OUT_F32, int FPC>
__global__ void __launch_bounds__(kThreads, 4) gemv_bf16_kernel(const GemvArgs a) {
  pdl_wait();
  constexpr int NT = 2;                 // 8-row column blocks per pass
  constexpr int U = 4;                  // 32-wide K chunks in flight per warp
  constexpr int WG = kWarps * 16 / FPC; // warps per 16-feature group (K split)
  __shared__ float red[kWarps][NT][128];
  __shared__ float wrs[2][NT * 8];      // routing weights of a pass's rows (EPI_SCALE)

  Seg sg;
  if (!resolve_id(a, sg)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int kw = warp % WG;             // this warp's K share within its group
  const int f0 = blockIdx.x * FPC + 16 * (warp / WG);
  const int K = a.K;

  const bf16* W = reinterpret_cast<const bf16*>(a.W) + sg.id * a.w_seg_stride + (int64_t)f0 * K;
  const bf16* wg = W + (int64_t)g * K + 8 * t4;
  const bf16* wg8 = W + (int64_t)(g + 8) * K + 8 * t4;
  const int nchunks = K >> 5;
  uint4 A0[U], A1[U];
  auto load_round = [&](int c) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cc = c + WG * u;
      if (cc < nchunks) {
        A0[u] = ldg_stream(wg + cc * 32);
        A1[u] = ldg_stream(wg8 + cc * 32);
      }
    }
  };
  // the first round of weight loads goes out before the row lookups and
  // gathers below, whose dependent loads would otherwise delay it
  load_round(kw);
  // dense products split their 16-row passes over grid.z (CTAs of one feature
  // tile run together, so the tile is read from HBM once; z < ceil(rows/16),
  // so no CTA returns here after loading); grouped ones loop
  if (!resolve_rows(a, a.offsets ? (1 << 30) : NT * 8, sg)) return;

  for (int p0 = 0, pi = 0; p0 < sg.nrows; p0 += NT * 8, ++pi) {
    const int prow = min(sg.nrows - p0, NT * 8);
    // the pass's routing weights, read after the K loop (double-buffered by
    // pass parity: the pass before the previous one has finished with them)
    if (EPI == EPI_SCALE && threadIdx.x < prow) wrs[pi & 1][threadIdx.x] = route_weight(a, sg.row0 + p0 + threadIdx.x);
    const bf16* xr[NT];
    bool xv[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int r = j * 8 + g;
      xv[j] = r < prow;
      int64_t row = 0;
      if (xv[j]) row = a.gather ? a.gather[sg.row0 + p0 + r] : (sg.row0 + p0 + r);
      xr[j] = reinterpret_cast<const bf16*>(a.X) + row * a.x_ld + 8 * t4;
    }
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    for (int c = kw; c < nchunks; c += WG * U) {
      if (p0 > 0 || c != kw) load_round(c);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c + WG * u;
        if (cc < nchunks) {
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            if (j * 8 < prow) {
              uint4 B = make_uint4(0, 0, 0, 0);
              if (xv[j]) B = ldg_keep(xr[j] + cc * 32);
              mma_bf16_16816(acc[j], A0[u].x, A1[u].x, A0[u].y, A1[u].y, B.x, B.y);
              mma_bf16_16816(acc[j], A0[u].z, A1[u].z, A0[u].w, A1[u].w, B.z, B.w);
            }
          }
        }
      }
    }

    // acc[j][0]: (feature g, row 2t), [1]: (g, 2t+1), [2]: (g+8, 2t), [3]: (g+8, 2t+1)
    if (p0 > 0) __syncthreads();      // previous pass has finished reading red
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      red[warp][j][g * 8 + 2 * t4] = acc[j][0];
      red[warp][j][g * 8 + 2 * t4 + 1] = acc[j][1];
      red[warp][j][(g + 8) * 8 + 2 * t4] = acc[j][2];
      red[warp][j][(g + 8) * 8 + 2 * t4 + 1] = acc[j][3];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < (FPC / 16) * NT * 128; o += kThreads) {
      const int gi = o / (NT * 128), j = (o >> 7) % NT, idx = o & 127;
      const int f = idx >> 3, r = j * 8 + (idx & 7);
      if (r < prow) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < WG; ++w) v += red[gi * WG + w][j][idx];
        epilogue_pre<EPI, OUT_F32, false>(a, sg.row0 + p0 + r, blockIdx.x * FPC + 16 * gi + f, v, 1.f,
                                          EPI == EPI_SCALE ? wrs[pi & 1][r] : 0.f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// NVFP4 weights (E2M1 values, one E4M3 scale per 16 K-elements, FP32 per-tensor
// scale), BF16 activations.  A warp streams 128-wide K chunks: 16 bytes of row
// g and of row g+8 per thread (32 values each) plus their two block scales.
// MMA k positions are the same consistent permutation as the BF16 kernel: MMA
// i of a chunk takes this thread's values 4i..4i+3 of each row and the
// matching activations.
// ---------------------------------------------------------------------------
// Each warp owns 16 features of the segment over the whole K, so partial sums
// never leave registers; the next chunk's weight bytes are requested before
// the current chunk is decoded.  Values are decoded by the hardware E2M1 and
// E4M3 conversions to FP16 and the block scale is applied by an exact FP16
// multiply (E2M1 x E4M3 spans 2^-10 .. 2688 with at most 6 significant bits);
// the MMA runs in FP16 with the BF16 activations converted to FP16, which is
// exact for magnitudes in [2^-14, 65504] (smaller ones keep FP16's subnormal
// precision); accumulation is FP32 and the per-tensor scale multiplies the
// FP32 result.

template <int EPI, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 3) gemv_nvfp4_kernel(const GemvArgs a) {
  pdl_wait();
  constexpr int NT = 2;
  Seg sg;
  if (!resolve_segment(a, 1 << 30, sg)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int K = a.K;
  const int64_t rowb = K / 2, rows_sf = K / 16;
  const int nchunks = K >> 7;

  for (int f0 = (blockIdx.x * kWarps + warp) * 16; f0 < a.N; f0 += gridDim.x * kWarps * 16) {
    const uint8_t* W = reinterpret_cast<const uint8_t*>(a.W) + sg.id * a.w_seg_stride + (int64_t)f0 * rowb;
    const uint8_t* SF = a.W_sf + sg.id * a.sf_seg_stride + (int64_t)f0 * rows_sf;
    const uint8_t* wg = W + (int64_t)g * rowb + 16 * t4;
    const uint8_t* wg8 = W + (int64_t)(g + 8) * rowb + 16 * t4;
    const uint8_t* sg0 = SF + (int64_t)g * rows_sf + 2 * t4;
    const uint8_t* sg8 = SF + (int64_t)(g + 8) * rows_sf + 2 * t4;

    for (int p0 = 0; p0 < sg.nrows; p0 += NT * 8) {
      const int prow = min(sg.nrows - p0, NT * 8);
      const bf16* xr[NT];
      bool xv[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int r = j * 8 + g;
        xv[j] = r < prow;
        int64_t row = 0;
        if (xv[j]) row = a.gather ? a.gather[sg.row0 + p0 + r] : (sg.row0 + p0 + r);
        xr[j] = reinterpret_cast<const bf16*>(a.X) + row * a.x_ld + 32 * t4;
      }
      float acc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

      uint4 nA0 = ldg_stream(wg), nA1 = ldg_stream(wg8);
      uint32_t nS0 = *reinterpret_cast<const uint16_t*>(sg0), nS1 = *reinterpret_cast<const uint16_t*>(sg8);
      for (int cc = 0; cc < nchunks; ++cc) {
        const uint4 A0 = nA0, A1 = nA1;
        const uint32_t S0 = nS0, S1 = nS1;
        if (cc + 1 < nchunks) {
          nA0 = ldg_stream(wg + (cc + 1) * 64);
          nA1 = ldg_stream(wg8 + (cc + 1) * 64);
          nS0 = *reinterpret_cast<const uint16_t*>(sg0 + (cc + 1) * 8);
          nS1 = *reinterpret_cast<const uint16_t*>(sg8 + (cc + 1) * 8);
        }
        // block scales (values 0..15 and 16..31 of each row's 32) as {s, s} pairs
        const uint32_t s0 = e4m3x2_to_f16x2(S0), s1 = e4m3x2_to_f16x2(S1);
        const uint32_t sc0[2] = {__byte_perm(s0, 0, 0x1010), __byte_perm(s0, 0, 0x3232)};
        const uint32_t sc1[2] = {__byte_perm(s1, 0, 0x1010), __byte_perm(s1, 0, 0x3232)};
        // fa[i]: A fragment of MMA i = this thread's values 4i..4i+3 of rows g and g+8
        uint32_t fa[8][4];
        const uint32_t w0[4] = {A0.x, A0.y, A0.z, A0.w};
        const uint32_t w1[4] = {A1.x, A1.y, A1.z, A1.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t p0v[4], p1v[4];
          e2m1x8_to_f16x2(w0[q], p0v);     // values 8q .. 8q+7 of row g
          e2m1x8_to_f16x2(w1[q], p1v);     // of row g+8
          const int h = q >> 1;
          fa[2 * q][0] = hmul2_f16(p0v[0], sc0[h]);
          fa[2 * q][2] = hmul2_f16(p0v[1], sc0[h]);
          fa[2 * q][1] = hmul2_f16(p1v[0], sc1[h]);
          fa[2 * q][3] = hmul2_f16(p1v[1], sc1[h]);
          fa[2 * q + 1][0] = hmul2_f16(p0v[2], sc0[h]);
          fa[2 * q + 1][2] = hmul2_f16(p0v[3], sc0[h]);
          fa[2 * q + 1][1] = hmul2_f16(p1v[2], sc1[h]);
          fa[2 * q + 1][3] = hmul2_f16(p1v[3], sc1[h]);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (j * 8 >= prow) continue;
          uint4 B[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) B[q] = xv[j] ? ldg_keep(xr[j] + cc * 128 + 8 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4& Bq = B[i >> 1];
            const uint32_t bb0 = bf16x2_to_f16x2((i & 1) ? Bq.z : Bq.x);
            const uint32_t bb1 = bf16x2_to_f16x2((i & 1) ? Bq.w : Bq.y);
            mma_f16_16816(acc[j], fa[i][0], fa[i][1], fa[i][2], fa[i][3], bb0, bb1);
          }
        }
      }
      // acc[j][0]: (feature g, row 2t), [1]: (g, 2t+1), [2]: (g+8, 2t), [3]: (g+8, 2t+1)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int r0 = j * 8 + 2 * t4;
        if (r0 < prow) {
          epilogue<EPI, OUT_F32, false>(a, sg.id, sg.row0 + p0 + r0, f0 + g, acc[j][0]);
          epilogue<EPI, OUT_F32, false>(a, sg.id, sg.row0 + p0 + r0, f0 + g + 8, acc[j][2]);
        }
        if (r0 + 1 < prow) {
          epilogue<EPI, OUT_F32, false>(a, sg.id, sg.row0 + p0 + r0 + 1, f0 + g, acc[j][1]);
          epilogue<EPI, OUT_F32, false>(a, sg.id, sg.row0 + p0 + r0 + 1, f0 + g + 8, acc[j][3]);
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// NVFP4 weights, bulk-copied (grouped decode products).  A CTA's 4 warps form
// groups of WPG warps; a group owns 16 features, a warp of the group every
// WPG-th 128-wide K chunk (WPG = 1 for K <= 1536, else 2), so a CTA covers
// 64 / WPG features.  Their packed rows (contiguous bytes) and block scales
// arrive in two cp.async.bulk copies on one mbarrier, so the whole tile is in
// flight at once whatever the register budget.  Each chunk is decoded exactly
// as above (hardware E2M1 / E4M3 conversion, exact FP16 scale multiply, same
// MMA k permutation) while the next chunk's activations load; a group's two
// partial sums are added in a fixed order.  Row passes of 16 re-read the tile
// from shared memory.  The activations may come as FP16 (the exact FP16 copy
// of BF16 values, made once per layer call) so that no CTA converts them
// again, and the up projection may store its ReLU^2 rows as FP16 copies of
// their BF16 values for the down projection to read the same way.
// ---------------------------------------------------------------------------
constexpr int kBulkWarps = 4;
constexpr int kBulkThreads = kBulkWarps * 32;
constexpr uint64_t kBulkWaitNs = 4000000000ull;
constexpr size_t kBulkSmemMax = 200 * 1024;

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

inline int nvfp4_wpg(int K) { return K <= 1536 ? 1 : 2; }

size_t nvfp4_bulk_smem(int K, int wpg) {
  const int rows = 16 * kBulkWarps / wpg;
  return (size_t)rows * (K / 2) + (size_t)rows * (K / 16) + (size_t)kBulkWarps * 2 * 128 * sizeof(float) + 16;
}

// an activation pair as the FP16 pair the MMA takes
template <bool XF16>
__device__ __forceinline__ uint32_t as_f16x2(uint32_t v) { return XF16 ? v : bf16x2_to_f16x2(v); }

// OUT: 0 = BF16, 1 = FP32, 2 = FP16 copy of the BF16 value; XF16: X is FP16
template <int EPI, int OUT, bool XF16, int WPG>
__global__ void __launch_bounds__(kBulkThreads) gemv_nvfp4_bulk_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) uint8_t bsm[];
  pdl_wait();
  constexpr int NT = 2;
  constexpr int ROWS = 16 * kBulkWarps / WPG;          // features of this CTA
  Seg sg;
  if (!resolve_id(a, sg)) return;       // grouped only: the copy needs the expert id alone
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int gi = warp / WPG, sub = warp % WPG;         // feature group, K share
  const int K = a.K;
  const int rowb = K / 2, rows_sf = K / 16;
  const int nchunks = K >> 7;
  const int fc = blockIdx.x * ROWS;                    // first feature of the CTA
  const int f0 = fc + 16 * gi;                         // first feature of this warp's group
  uint8_t* ws = bsm;                                   // [ROWS][K/2] packed values
  uint8_t* ss = bsm + ROWS * rowb;                     // [ROWS][K/16] E4M3 scales
  float* red = reinterpret_cast<float*>(ss + ROWS * rows_sf);   // [warps][NT][4][32] (WPG 2)
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + kBulkWarps * NT * 128);
  const uint32_t b = smem_u32(bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t wbytes = (uint32_t)ROWS * rowb, sbytes = (uint32_t)ROWS * rows_sf;
    mbar_expect_tx(b, wbytes + sbytes);
    bulk_g2s(smem_u32(ws), reinterpret_cast<const uint8_t*>(a.W) + sg.id * a.w_seg_stride + (int64_t)fc * rowb, wbytes,
             b);
    bulk_g2s(smem_u32(ss), a.W_sf + sg.id * a.sf_seg_stride + (int64_t)fc * rows_sf, sbytes, b);
  }
  // the rows, the segment's per-tensor scale and the rows' routing weights
  // load while the weight tile is in flight (an active expert has rows, so no
  // CTA leaves here with its copy outstanding)
  resolve_rows(a, 1 << 30, sg);
  const float gs = a.W_gs ? a.W_gs[sg.id] : 1.f;
  __shared__ float wrs[1][16];
  if (EPI == EPI_SCALE && threadIdx.x < min(sg.nrows, 16)) wrs[0][threadIdx.x] = route_weight(a, sg.row0 + threadIdx.x);
  {
    // the first pass's activation rows are pulled into L1 while the weight
    // tile is in flight: every warp reads all of them, chunk by chunk, and a
    // load that went to L2 each chunk would stall the chunk loop
    const int lines = K / 64;                          // 128-byte lines of a row (2-byte values)
    const int n = min(sg.nrows, 16) * lines;
    for (int i = threadIdx.x; i < n; i += kBulkThreads) {
      const int r = i / lines;
      const int64_t row = a.gather ? a.gather[sg.row0 + r] : (sg.row0 + r);
      prefetch_l1(reinterpret_cast<const uint16_t*>(a.X) + row * a.x_ld + (i - r * lines) * 64);
    }
  }
  __syncthreads();
  bool ok = mbar_try(b, 0);
  if (!ok) {
    const uint64_t t0 = globaltimer();
    while (!(ok = mbar_try(b, 0)) && globaltimer() - t0 < kBulkWaitNs) {
    }
  }
  if (!ok) {
    // the copies never completed: report, and keep the CTA alive (bounded)
    // while they may still land in its shared memory
    if (threadIdx.x == 0) {
      set_error(a.err, MOE_DEVERR_TIMEOUT);
      const uint64_t t0 = globaltimer();
      while (!mbar_try(b, 0) && globaltimer() - t0 < kBulkWaitNs) {
      }
    }
    return;
  }
  const uint8_t* wrow = ws + (16 * gi) * rowb;
  const uint8_t* srow = ss + (16 * gi) * rows_sf;

  for (int p0 = 0; p0 < sg.nrows; p0 += NT * 8) {
    const int prow = min(sg.nrows - p0, NT * 8);
    if (p0 > 0) {
      // every warp has finished the previous pass (its epilogue read wrs, its
      // partial sums were read from red)
      __syncthreads();
      if (EPI == EPI_SCALE && threadIdx.x < prow) wrs[0][threadIdx.x] = route_weight(a, sg.row0 + p0 + threadIdx.x);
      __syncthreads();
    }
    // activation rows of the pass (a lane past the last row loads nothing)
    const uint16_t* xr[NT];
    bool xv[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      xv[j] = j * 8 + g < prow;
      const int64_t row = !xv[j] ? 0 : a.gather ? a.gather[sg.row0 + p0 + j * 8 + g] : (sg.row0 + p0 + j * 8 + g);
      xr[j] = reinterpret_cast<const uint16_t*>(a.X) + row * a.x_ld + 32 * t4;
    }
    const bool two = prow > 8;
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    // activations of the first chunk; later chunks load one chunk ahead
    uint4 B0[4], B1[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) B0[q] = B1[q] = make_uint4(0, 0, 0, 0);
    if (sub < nchunks) {
#pragma unroll
      for (int q = 0; q < 4; ++q) B0[q] = xv[0] ? ldg_keep(xr[0] + sub * 128 + 8 * q) : make_uint4(0, 0, 0, 0);
      if (two) {
#pragma unroll
        for (int q = 0; q < 4; ++q) B1[q] = xv[1] ? ldg_keep(xr[1] + sub * 128 + 8 * q) : make_uint4(0, 0, 0, 0);
      }
    }
    for (int cc = sub; cc < nchunks; cc += WPG) {
      const int cn = cc + WPG;
      uint4 N0[4], N1[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) N0[q] = N1[q] = make_uint4(0, 0, 0, 0);
      if (cn < nchunks) {
#pragma unroll
        for (int q = 0; q < 4; ++q) N0[q] = xv[0] ? ldg_keep(xr[0] + cn * 128 + 8 * q) : make_uint4(0, 0, 0, 0);
        if (two) {
#pragma unroll
          for (int q = 0; q < 4; ++q) N1[q] = xv[1] ? ldg_keep(xr[1] + cn * 128 + 8 * q) : make_uint4(0, 0, 0, 0);
        }
      }
      const uint4 A0 = *reinterpret_cast<const uint4*>(wrow + g * rowb + cc * 64 + 16 * t4);
      const uint4 A1 = *reinterpret_cast<const uint4*>(wrow + (g + 8) * rowb + cc * 64 + 16 * t4);
      const uint32_t S0 = *reinterpret_cast<const uint16_t*>(srow + g * rows_sf + cc * 8 + 2 * t4);
      const uint32_t S1 = *reinterpret_cast<const uint16_t*>(srow + (g + 8) * rows_sf + cc * 8 + 2 * t4);
      const uint32_t s0 = e4m3x2_to_f16x2(S0), s1 = e4m3x2_to_f16x2(S1);
      const uint32_t sc0[2] = {__byte_perm(s0, 0, 0x1010), __byte_perm(s0, 0, 0x3232)};
      const uint32_t sc1[2] = {__byte_perm(s1, 0, 0x1010), __byte_perm(s1, 0, 0x3232)};
      const uint32_t w0[4] = {A0.x, A0.y, A0.z, A0.w};
      const uint32_t w1[4] = {A1.x, A1.y, A1.z, A1.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t p0v[4], p1v[4];
        e2m1x8_to_f16x2(w0[q], p0v);     // values 8q .. 8q+7 of row g
        e2m1x8_to_f16x2(w1[q], p1v);     // of row g+8
        const int h = q >> 1;
        // MMA 2q: values 8q..8q+3, MMA 2q+1: 8q+4..8q+7 (this thread's k slots)
        const uint32_t fa0[4] = {hmul2_f16(p0v[0], sc0[h]), hmul2_f16(p1v[0], sc1[h]), hmul2_f16(p0v[1], sc0[h]),
                                 hmul2_f16(p1v[1], sc1[h])};
        const uint32_t fa1[4] = {hmul2_f16(p0v[2], sc0[h]), hmul2_f16(p1v[2], sc1[h]), hmul2_f16(p0v[3], sc0[h]),
                                 hmul2_f16(p1v[3], sc1[h])};
        mma_f16_16816(acc[0], fa0[0], fa0[1], fa0[2], fa0[3], as_f16x2<XF16>(B0[q].x), as_f16x2<XF16>(B0[q].y));
        mma_f16_16816(acc[0], fa1[0], fa1[1], fa1[2], fa1[3], as_f16x2<XF16>(B0[q].z), as_f16x2<XF16>(B0[q].w));
        if (two) {
          mma_f16_16816(acc[1], fa0[0], fa0[1], fa0[2], fa0[3], as_f16x2<XF16>(B1[q].x), as_f16x2<XF16>(B1[q].y));
          mma_f16_16816(acc[1], fa1[0], fa1[1], fa1[2], fa1[3], as_f16x2<XF16>(B1[q].z), as_f16x2<XF16>(B1[q].w));
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        B0[q] = N0[q];
        B1[q] = N1[q];
      }
    }

    // acc[j][0]: (feature g, row 2t), [1]: (g, 2t+1), [2]: (g+8, 2t), [3]: (g+8, 2t+1)
    if (WPG > 1) {
      if (sub != 0) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) red[((warp * NT + j) * 4 + i) * 32 + lane] = acc[j][i];
      }
      __syncthreads();
    }
    if (sub == 0) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float v[4] = {acc[j][0], acc[j][1], acc[j][2], acc[j][3]};
#pragma unroll
        for (int w = 1; w < WPG; ++w)
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] += red[(((warp + w) * NT + j) * 4 + i) * 32 + lane];
        const int r0 = j * 8 + 2 * t4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = r0 + (i & 1), f = f0 + g + (i >> 1) * 8;
          if (r < prow) {
            const float wr = EPI == EPI_SCALE ? wrs[0][r] : 0.f;
            if (OUT == 2) epilogue_pre_f16<EPI>(a, sg.row0 + p0 + r, f, v[i], gs, wr);
            else epilogue_pre<EPI, OUT == 1, false>(a, sg.row0 + p0 + r, f, v[i], gs, wr);
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// FP32 weights and activations (small FP32 layers): plain FMA dot products.
// A CTA owns 64 features of one segment and up to 64 rows.
// ---------------------------------------------------------------------------
template <int EPI>
__global__ void __launch_bounds__(kThreads) gemv_f32_kernel(const GemvArgs a) {
  pdl_wait();
  Seg sg;
  if (!resolve_segment(a, 64, sg)) return;
  const int fl = threadIdx.x & 63, rg = threadIdx.x >> 6;
  const int f = blockIdx.x * 64 + fl;
  if (f >= a.N) return;
  const float* w = reinterpret_cast<const float*>(a.W) + sg.id * a.w_seg_stride + (int64_t)f * a.K;
  for (int r = rg; r < sg.nrows; r += 4) {
    const int64_t row = a.gather ? a.gather[sg.row0 + r] : (sg.row0 + r);
    const float* x = reinterpret_cast<const float*>(a.X) + row * a.x_ld;
    float acc = 0.f;
    for (int k = 0; k < a.K; k += 4) {
      const float4 wv = *reinterpret_cast<const float4*>(w + k);
      const float4 xv = *reinterpret_cast<const float4*>(x + k);
      acc = fmaf(wv.x, xv.x, acc);
      acc = fmaf(wv.y, xv.y, acc);
      acc = fmaf(wv.z, xv.z, acc);
      acc = fmaf(wv.w, xv.w, acc);
    }
    epilogue<EPI, true, true>(a, sg.id, sg.row0 + r, f, acc);
  }
}

// the NVFP4 bulk GEMV's shared-memory limit for both warp splits
template <int EPI, int OUT, bool XF16>
cudaError_t bulk_attr() {
  cudaError_t e = cudaFuncSetAttribute((const void*)gemv_nvfp4_bulk_kernel<EPI, OUT, XF16, 1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmemMax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute((const void*)gemv_nvfp4_bulk_kernel<EPI, OUT, XF16, 2>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmemMax);
}

// FP16 copy of BF16 activations, 8 values per thread; a value beyond FP16's
// range sets MOE_DEVERR_RANGE
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* x, int64_t n8, uint4* out, int32_t* err) {
  pdl_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 v = x[i];
  if (err && bf16x4_beyond_f16(v)) set_error(err, MOE_DEVERR_RANGE);
  out[i] = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
}

// 32 features per CTA for rows of at most 2048 values (a 16-feature CTA would
// stream under 64 KB of weights), 16 otherwise
template <int EPI, bool OUT_F32>
cudaError_t pick_nt(const GemvArgs& a, int max_rows, int segs, cudaStream_t s) {
  const unsigned z = a.offsets ? 1u : (unsigned)ceil_div(max_rows, 16);
  if (a.K <= 2048 && a.N % 32 == 0) {
    launch_k(gemv_bf16_kernel<EPI, OUT_F32, 32>, dim3(a.N / 32, segs, z), kThreads, 0, s, a);
    return cudaGetLastError();
  }
  launch_k(gemv_bf16_kernel<EPI, OUT_F32, 16>, dim3(a.N / 16, segs, z), kThreads, 0, s, a);
  return cudaGetLastError();
}

}  // namespace

bool gemv_nvfp4_streams(const GemvArgs& a) {
  const int wpg = nvfp4_wpg(a.K);
  return a.offsets && a.K % 128 == 0 && a.N % (64 / wpg) == 0 && nvfp4_bulk_smem(a.K, wpg) <= kBulkSmemMax &&
         !(reinterpret_cast<uintptr_t>(a.W) & 15) && !(reinterpret_cast<uintptr_t>(a.W_sf) & 15);
}

cudaError_t launch_bf16_to_f16(const void* x, int64_t n, void* out, cudaStream_t s, int32_t* err) {
  if (n <= 0) return cudaSuccess;
  const int64_t v = n / 8;
  launch_k(bf16_to_f16_kernel, dim3((unsigned)ceil_div(v, 256)), 256, 0, s, reinterpret_cast<const uint4*>(x), v,
           reinterpret_cast<uint4*>(out), err);
  return cudaGetLastError();
}

cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int act, int epi, bool out_f32, int max_rows,
                        int segs, cudaStream_t s) {
  if (max_rows <= 0 || segs <= 0) return cudaSuccess;
  if (wfmt == WF_F32) {
    dim3 grid((unsigned)ceil_div(a.N, 64), segs, (unsigned)ceil_div(max_rows, 64));
    switch (epi) {
      case EPI_RELU2: launch_k(gemv_f32_kernel<EPI_RELU2>, grid, kThreads, 0, s, a); break;
      case EPI_SCALE: launch_k(gemv_f32_kernel<EPI_SCALE>, grid, kThreads, 0, s, a); break;
      case EPI_STORE: launch_k(gemv_f32_kernel<EPI_STORE>, grid, kThreads, 0, s, a); break;
      default: launch_k(gemv_f32_kernel<EPI_ADD>, grid, kThreads, 0, s, a); break;
    }
    return cudaGetLastError();
  }
  if (wfmt == WF_NVFP4 && act == MOE_DT_BF16 && gemv_nvfp4_streams(a)) {
    // one CTA per 64 / WPG features of each active segment, weight tile bulk-copied
    const int wpg = nvfp4_wpg(a.K);
    const size_t smem = nvfp4_bulk_smem(a.K, wpg);
    void (*k)(GemvArgs) = nullptr;
#define MOE_NVK(E_, O_, X_) (wpg == 1 ? gemv_nvfp4_bulk_kernel<E_, O_, X_, 1> : gemv_nvfp4_bulk_kernel<E_, O_, X_, 2>)
    if (epi == EPI_RELU2 && !out_f32) {
      k = a.out_f16 ? (a.x_f16 ? MOE_NVK(EPI_RELU2, 2, true) : MOE_NVK(EPI_RELU2, 2, false))
                    : (a.x_f16 ? MOE_NVK(EPI_RELU2, 0, true) : MOE_NVK(EPI_RELU2, 0, false));
    } else if (epi == EPI_SCALE && out_f32 && !a.out_f16) {
      k = a.x_f16 ? MOE_NVK(EPI_SCALE, 1, true) : MOE_NVK(EPI_SCALE, 1, false);
    } else {
      return cudaErrorNotSupported;
    }
#undef MOE_NVK
    // every instantiation's shared-memory limit, set once per device
    static PerDeviceOnce attr_once;
    const cudaError_t attr = attr_once.run([](int&) {
      for (cudaError_t e : {bulk_attr<EPI_RELU2, 0, false>(), bulk_attr<EPI_RELU2, 0, true>(),
                            bulk_attr<EPI_RELU2, 2, false>(), bulk_attr<EPI_RELU2, 2, true>(),
                            bulk_attr<EPI_SCALE, 1, false>(), bulk_attr<EPI_SCALE, 1, true>()})
        if (e != cudaSuccess) return e;
      return cudaSuccess;
    });
    if (attr != cudaSuccess) return attr;
    return launch_k(k, dim3((unsigned)(a.N / (64 / wpg)), segs, 1), kBulkThreads, smem, s, a);
  }
  if (a.x_f16 || a.out_f16) return cudaErrorNotSupported;
  if (wfmt == WF_NVFP4 && act == MOE_DT_BF16) {
    // one warp per 16 features: a CTA's 8 warps cover 128 features
    dim3 grid((unsigned)ceil_div(a.N / 16, kWarps), segs, 1);
    switch (epi) {
      case EPI_RELU2: launch_k(gemv_nvfp4_kernel<EPI_RELU2, false>, grid, kThreads, 0, s, a); break;
      case EPI_SCALE: launch_k(gemv_nvfp4_kernel<EPI_SCALE, true>, grid, kThreads, 0, s, a); break;
      default: return cudaErrorNotSupported;
    }
    return cudaGetLastError();
  }
  if (wfmt != WF_BF16 || act != MOE_DT_BF16) return cudaErrorNotSupported;
  switch (epi) {
    case EPI_RELU2: return pick_nt<EPI_RELU2, false>(a, max_rows, segs, s);
    case EPI_SCALE: return pick_nt<EPI_SCALE, true>(a, max_rows, segs, s);
    case EPI_STORE:
      return out_f32 ? pick_nt<EPI_STORE, true>(a, max_rows, segs, s)
                     : pick_nt<EPI_STORE, false>(a, max_rows, segs, s);
    default:
      return out_f32 ? pick_nt<EPI_ADD, true>(a, max_rows, segs, s)
                     : pick_nt<EPI_ADD, false>(a, max_rows, segs, s);
  }
}

}  // namespace moe
