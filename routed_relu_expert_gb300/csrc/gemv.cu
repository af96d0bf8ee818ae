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

#include <algorithm>

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct Seg {
  int id, row0, nrows;
};

__device__ __forceinline__ bool resolve_segment(const GemvArgs& a, int rows_per_cta, Seg& s) {
  if (a.offsets) {
    const int j = blockIdx.y;
    if (j >= a.hdr->n_active) return false;
    s.id = a.active[j];
    s.row0 = a.offsets[s.id];
    s.nrows = a.offsets[s.id + 1] - s.row0;
  } else {
    s.id = 0;
    s.row0 = 0;
    s.nrows = a.dense_rows;
  }
  const int rb = blockIdx.z * rows_per_cta;
  if (rb >= s.nrows) return false;
  s.row0 += rb;
  s.nrows = min(s.nrows - rb, rows_per_cta);
  return true;
}

// ---------------------------------------------------------------------------
// BF16 weights, BF16 activations.  A CTA handles its segment's rows in passes
// of 16 (two 8-row MMA column blocks); a second pass finds the CTA's weight
// tile still in L2, so HBM streams each weight once while registers stay low.
// ---------------------------------------------------------------------------
template <int EPI, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 4) gemv_bf16_kernel(const GemvArgs a) {
  constexpr int NT = 2;                 // 8-row column blocks per pass
  constexpr int U = 4;                  // 32-wide K chunks in flight per warp
  __shared__ float red[kWarps][NT][128];

  Seg sg;
  if (!resolve_segment(a, 1 << 30, sg)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int f0 = blockIdx.x * 16;
  const int K = a.K;

  const bf16* W = reinterpret_cast<const bf16*>(a.W) + sg.id * a.w_seg_stride + (int64_t)f0 * K;
  const bf16* wg = W + (int64_t)g * K + 8 * t4;
  const bf16* wg8 = W + (int64_t)(g + 8) * K + 8 * t4;
  const int nchunks = K >> 5;

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
      xr[j] = reinterpret_cast<const bf16*>(a.X) + row * a.x_ld + 8 * t4;
    }
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    for (int c = warp; c < nchunks; c += kWarps * U) {
      uint4 A0[U], A1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c + kWarps * u;
        if (cc < nchunks) {
          A0[u] = ldg_stream(wg + cc * 32);
          A1[u] = ldg_stream(wg8 + cc * 32);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c + kWarps * u;
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
    for (int o = threadIdx.x; o < NT * 128; o += kThreads) {
      const int j = o >> 7, idx = o & 127;
      const int f = idx >> 3, r = j * 8 + (idx & 7);
      if (r < prow) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[w][j][idx];
        epilogue<EPI, OUT_F32, false>(a, sg.id, sg.row0 + p0 + r, f0 + f, v);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// NVFP4 weights (E2M1 values, one E4M3 scale per 16 K-elements, FP32 per-tensor
// scale), BF16 activations.  A warp streams 128-wide K chunks: 16 bytes of row
// g and of row g+8 per thread (32 values each) plus their two block scales.
// Each byte (two values) becomes a BF16 pair through a 256-entry table kept in
// 32 bank-private copies, then one exact BF16 multiply applies the block
// scale (E2M1 x E4M3 needs at most 6 significant bits); the per-tensor scale
// multiplies the FP32 result in the epilogue.  MMA k positions are the same
// consistent permutation trick as the BF16 kernel: MMA i of a chunk takes this
// thread's values 4i..4i+3 of each row and the matching activations.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e2m1_pair_bf16(uint32_t byte) {
  const uint16_t mag[8] = {0x0000, 0x3F00, 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0};
  const uint32_t lo = mag[byte & 7] | ((byte & 8u) << 12);
  const uint32_t hi = mag[(byte >> 4) & 7] | (((byte >> 7) & 1u) << 15);
  return lo | (hi << 16);
}

// E4M3 byte -> FP32: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
// field 0 is subnormal (M * 2^-9); 0x7F / 0xFF are NaN.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t s = (b & 0x80u) << 24, E = (b >> 3) & 15u, M = b & 7u;
  if (E == 15u && M == 7u) return __uint_as_float(0x7FC00000u | s);
  if (E == 0u) return __uint_as_float(s | __float_as_uint((float)M * 0.001953125f));
  return __uint_as_float(s | ((E + 120u) << 23) | (M << 20));
}

template <int EPI, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 3) gemv_nvfp4_kernel(const GemvArgs a) {
  constexpr int NT = 2;
  constexpr int U = 2;
  __shared__ uint32_t lut[256 * 32];
  __shared__ float red[kWarps][NT][128];
  for (int i = threadIdx.x; i < 256 * 32; i += kThreads) lut[i] = e2m1_pair_bf16((uint32_t)(i >> 5));
  __syncthreads();

  Seg sg;
  if (!resolve_segment(a, 1 << 30, sg)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int f0 = blockIdx.x * 16;
  const int K = a.K;
  const int64_t rowb = K / 2, rows_sf = K / 16;
  const uint8_t* W = reinterpret_cast<const uint8_t*>(a.W) + sg.id * a.w_seg_stride + (int64_t)f0 * rowb;
  const uint8_t* SF = a.W_sf + sg.id * a.sf_seg_stride + (int64_t)f0 * rows_sf;
  const uint8_t* wg = W + (int64_t)g * rowb + 16 * t4;
  const uint8_t* wg8 = W + (int64_t)(g + 8) * rowb + 16 * t4;
  const uint8_t* sg0 = SF + (int64_t)g * rows_sf + 2 * t4;
  const uint8_t* sg8 = SF + (int64_t)(g + 8) * rows_sf + 2 * t4;
  const uint32_t* lutl = lut + lane;
  const int nchunks = K >> 7;

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

    for (int c = warp; c < nchunks; c += kWarps * U) {
      uint4 A0[U], A1[U];
      uint32_t S0[U], S1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c + kWarps * u;
        if (cc < nchunks) {
          A0[u] = ldg_stream(wg + cc * 64);
          A1[u] = ldg_stream(wg8 + cc * 64);
          S0[u] = *reinterpret_cast<const uint16_t*>(sg0 + cc * 8);
          S1[u] = *reinterpret_cast<const uint16_t*>(sg8 + cc * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c + kWarps * u;
        if (cc >= nchunks) continue;
        // block scales of rows g / g+8 for values 0..15 and 16..31, as BF16 pairs
        __nv_bfloat162 sc0[2], sc1[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          sc0[h] = __float2bfloat162_rn(e4m3_to_f32((S0[u] >> (8 * h)) & 0xFFu));
          sc1[h] = __float2bfloat162_rn(e4m3_to_f32((S1[u] >> (8 * h)) & 0xFFu));
        }
        const uint32_t w0[4] = {A0[u].x, A0[u].y, A0[u].z, A0[u].w};
        const uint32_t w1[4] = {A1[u].x, A1[u].y, A1[u].z, A1[u].w};
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (j * 8 >= prow) continue;
          uint4 B[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) B[q] = xv[j] ? ldg_keep(xr[j] + cc * 128 + 8 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // bytes 2i, 2i+1 of this thread's 16 bytes of each row: values 4i .. 4i+3
            const int wi = i >> 1, sh = (i & 1) * 16;
            const uint32_t b0 = (w0[wi] >> sh) & 0xFFu, b1 = (w0[wi] >> (sh + 8)) & 0xFFu;
            const uint32_t c0 = (w1[wi] >> sh) & 0xFFu, c1 = (w1[wi] >> (sh + 8)) & 0xFFu;
            const int h = i >> 2;
            __nv_bfloat162 v;
            uint32_t a0, a1, a2, a3;
            v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&lutl[b0 << 5]), sc0[h]);
            a0 = *reinterpret_cast<uint32_t*>(&v);
            v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&lutl[b1 << 5]), sc0[h]);
            a2 = *reinterpret_cast<uint32_t*>(&v);
            v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&lutl[c0 << 5]), sc1[h]);
            a1 = *reinterpret_cast<uint32_t*>(&v);
            v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&lutl[c1 << 5]), sc1[h]);
            a3 = *reinterpret_cast<uint32_t*>(&v);
            const uint4& Bq = B[i >> 1];
            const uint32_t bb0 = (i & 1) ? Bq.z : Bq.x, bb1 = (i & 1) ? Bq.w : Bq.y;
            mma_bf16_16816(acc[j], a0, a1, a2, a3, bb0, bb1);
          }
        }
      }
    }

    if (p0 > 0) __syncthreads();
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      red[warp][j][g * 8 + 2 * t4] = acc[j][0];
      red[warp][j][g * 8 + 2 * t4 + 1] = acc[j][1];
      red[warp][j][(g + 8) * 8 + 2 * t4] = acc[j][2];
      red[warp][j][(g + 8) * 8 + 2 * t4 + 1] = acc[j][3];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < NT * 128; o += kThreads) {
      const int j = o >> 7, idx = o & 127;
      const int f = idx >> 3, r = j * 8 + (idx & 7);
      if (r < prow) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[w][j][idx];
        epilogue<EPI, OUT_F32, false>(a, sg.id, sg.row0 + p0 + r, f0 + f, v);
      }
    }
  }
}

// NVFP4 -> BF16 of whole matrices (for the tensor-core path): each output is
// E2M1 * E4M3 (exact in BF16); the per-tensor scale stays for the epilogue.
__global__ void dequant_nvfp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int64_t n_bytes,
                                     uint32_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_bytes; i += (int64_t)gridDim.x * blockDim.x) {
    const float s = e4m3_to_f32(sf[i >> 3]);
    const uint32_t p = e2m1_pair_bf16(q[i]);
    const float lo = __uint_as_float(p << 16) * s, hi = __uint_as_float(p & 0xFFFF0000u) * s;
    out[i] = (uint32_t)bf16_bits(lo) | ((uint32_t)bf16_bits(hi) << 16);
  }
}

// ---------------------------------------------------------------------------
// FP32 weights and activations (small FP32 layers): plain FMA dot products.
// A CTA owns 64 features of one segment and up to 64 rows.
// ---------------------------------------------------------------------------
template <int EPI>
__global__ void __launch_bounds__(kThreads) gemv_f32_kernel(const GemvArgs a) {
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

template <int EPI, bool OUT_F32>
cudaError_t pick_nt(const GemvArgs& a, int max_rows, int segs, cudaStream_t s) {
  (void)max_rows;
  dim3 grid(a.N / 16, segs, 1);
  gemv_bf16_kernel<EPI, OUT_F32><<<grid, kThreads, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant_nvfp4(const uint8_t* q, const uint8_t* sf, int64_t n_values, void* out, cudaStream_t s) {
  const int64_t n_bytes = n_values / 2;
  if (n_bytes <= 0) return cudaSuccess;
  dequant_nvfp4_kernel<<<(unsigned)std::min<int64_t>(ceil_div(n_bytes, 256), 16384), 256, 0, s>>>(
      q, sf, n_bytes, reinterpret_cast<uint32_t*>(out));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int act, int epi, bool out_f32, int max_rows,
                        int segs, cudaStream_t s) {
  if (max_rows <= 0 || segs <= 0) return cudaSuccess;
  if (wfmt == WF_F32) {
    dim3 grid((unsigned)ceil_div(a.N, 64), segs, (unsigned)ceil_div(max_rows, 64));
    switch (epi) {
      case EPI_RELU2: gemv_f32_kernel<EPI_RELU2><<<grid, kThreads, 0, s>>>(a); break;
      case EPI_SCALE: gemv_f32_kernel<EPI_SCALE><<<grid, kThreads, 0, s>>>(a); break;
      case EPI_STORE: gemv_f32_kernel<EPI_STORE><<<grid, kThreads, 0, s>>>(a); break;
      default: gemv_f32_kernel<EPI_ADD><<<grid, kThreads, 0, s>>>(a); break;
    }
    count_launches(1);
    return cudaGetLastError();
  }
  if (wfmt == WF_NVFP4 && act == MOE_DT_BF16) {
    dim3 grid(a.N / 16, segs, 1);
    switch (epi) {
      case EPI_RELU2: gemv_nvfp4_kernel<EPI_RELU2, false><<<grid, kThreads, 0, s>>>(a); break;
      case EPI_SCALE: gemv_nvfp4_kernel<EPI_SCALE, true><<<grid, kThreads, 0, s>>>(a); break;
      default: return cudaErrorNotSupported;
    }
    count_launches(1);
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
