// Backward of the routed ReLU^2 layer (page "M6.1 Routed Capacity", section
// 0x06F "Single-Device Forward And Backward Integration Contract": the
// forward's route tensors are the coordinates of the backward; the combine's
// backward is a broadcast (dU = w dY) and a dot product (q = <dY, U>); the
// gather's adjoint is a scatter-add; the router and expert paths meet again at
// the input, and the block's residual is a third path).  The gate here is
// sigmoid -> normalise -> scale (page "Nemotron Is Not One Circuit", section
// "The Router Is A Deterministic Algorithm"), not the page's selected softmax.
//
// Every product of the backward is one grouped BF16 GEMM with FP32
// accumulation, C[m, n] = sum_k A[m, k] B[k, n], in one of two groupings:
//  - rows by expert (GM_ROWS): the packed rows of expert e times expert e's
//    weight matrix (dh = dU W_down,e; dx = da W_up,e), or one dense product;
//  - K by expert (GM_KSEG): a weight gradient, dW_e += A_e^T B_e with K over
//    the packed rows of expert e (or over all tokens for a dense matrix).
// A is read row-major ([m][k]) or transposed ([k][m]); B is always [k][n] (the
// stored [out, in] weights taken as [k][n]); each CTA stages 64 x 32 and
// 32 x 64 tiles in shared memory with cp.async (double-buffered) and feeds
// m16n8k16 MMAs through ldmatrix (.trans where the tile is k-major).  The
// products are small next to the forward's (a training step's backward
// streams each touched weight matrix about twice), so this mma.sync kernel is
// the plain tensor-core path, not the forward's tcgen05 pipeline.  Each C
// tile belongs to one CTA: sums run in a fixed order and the result does not
// depend on scheduling.
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 64, BN = 64, BK = 32;
constexpr int kGThreads = 128;
constexpr int A_LD = BK + 8;      // [m][k] tile row stride (elements)
constexpr int AT_LD = BM + 8;     // [k][m] tile row stride
constexpr int B_LD = BN + 8;      // [k][n] tile row stride

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;     // 0: the 16 bytes are zero-filled, nothing is read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// rows [r0, r1) of this CTA's segment (GM_ROWS) or its K range (GM_KSEG), and
// the segment's expert id; false: nothing to do
__device__ __forceinline__ bool gemm_segment(const GemmArgs& g, int j, int& e, int& r0, int& r1) {
  if (!g.offsets) {
    e = 0;
    r0 = 0;
    r1 = g.dense_rows;
    return r1 > 0;
  }
  if (j >= g.hdr->n_active) return false;
  e = g.active[j];
  r0 = g.offsets[e];
  r1 = g.offsets[e + 1];
  return r1 > r0;
}

// GM_ROWS over expert segments: 64-row tile tau of the flattened list (tile
// prefix over the active segments) -> segment j and its rows [r0, r1), tile
// rows m0..
__device__ __forceinline__ bool gemm_row_tile(const GemmArgs& g, int tau, int& e, int& m0, int& r1) {
  const int na = g.hdr->n_active;
  if (tau >= g.tprefix[na]) return false;
  int lo = 0, hi = na - 1;                 // last j with tprefix[j] <= tau
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (g.tprefix[mid] <= tau) lo = mid; else hi = mid - 1;
  }
  e = g.active[lo];
  m0 = g.offsets[e] + (tau - g.tprefix[lo]) * 64;
  r1 = g.offsets[e + 1];
  return m0 < r1;
}

template <bool A_T, int EPI>
__global__ void __launch_bounds__(kGThreads) gemm_bwd_kernel(const GemmArgs g) {
  pdl_wait();
  __shared__ __align__(128) bf16 As[2][A_T ? BK * AT_LD : BM * A_LD];
  __shared__ __align__(128) bf16 Bs[2][BK * B_LD];
  const bool kseg = g.mode == GM_KSEG;
  // output tile: rows m0.., cols n0..; K range [k0, k1)
  int e, m0, mend, k0, k1;
  if (kseg) {
    if (!gemm_segment(g, (int)blockIdx.z, e, k0, k1)) return;
    m0 = blockIdx.y * BM;
    mend = g.M;
  } else if (g.offsets) {
    if (!gemm_row_tile(g, (int)blockIdx.y, e, m0, mend)) return;
    k0 = 0;
    k1 = g.K;
  } else {
    e = 0;
    m0 = blockIdx.y * BM;
    mend = g.dense_rows;
    if (m0 >= mend) return;
    k0 = 0;
    k1 = g.K;
  }
  const int n0 = blockIdx.x * BN;
  const bf16* Bseg = g.B + (int64_t)e * g.b_seg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;

  auto load = [&](int st, int kt) {
    // A: 256 16-byte chunks
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int q = tid + c * kGThreads;
      if (!A_T) {
        const int r = q >> 2, kc = (q & 3) * 8;        // row m0 + r, k kt + kc
        const int m = m0 + r;
        const bool ok = m < mend;
        const int64_t row = ok ? (g.a_gather ? g.a_gather[m] : m) : 0;
        cp_async16(smem_u32(&As[st][r * A_LD + kc]), g.A + row * g.lda + kt + kc, ok);
      } else {
        const int r = q >> 3, mc = (q & 7) * 8;        // k row kt + r, m m0 + mc
        const int k = kt + r;
        const bool ok = k < k1 && m0 + mc < g.M;
        cp_async16(smem_u32(&As[st][r * AT_LD + mc]), g.A + (ok ? (int64_t)k * g.lda + m0 + mc : 0), ok);
      }
    }
    // B: 32 k rows x 64 n, 256 chunks
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int q = tid + c * kGThreads;
      const int r = q >> 3, nc = (q & 7) * 8;
      const int k = kt + r;
      const bool ok = k < k1 && n0 + nc < g.N;
      int64_t krow = 0;
      if (ok) krow = g.b_gather ? g.b_gather[k] : k;
      cp_async16(smem_u32(&Bs[st][r * B_LD + nc]), Bseg + (ok ? krow * g.ldb + n0 + nc : 0), ok);
    }
    cp_async_commit();
  };

  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

  const int ntiles = (k1 - k0 + BK - 1) / BK;
  if (ntiles > 0) load(0, k0);
  for (int it = 0; it < ntiles; ++it) {
    const int st = it & 1;
    if (it + 1 < ntiles) {
      load(st ^ 1, k0 + (it + 1) * BK);
      cp_async_wait1();
    } else {
      cp_async_wait0();
    }
    __syncthreads();
#pragma unroll
    for (int ks = 0; ks < BK; ks += 16) {
      uint32_t a[2][4], b[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        if (!A_T) {
          const int r = wm + mi * 16 + (lane & 15), c = ks + (lane >> 4) * 8;
          ldsm_x4(smem_u32(&As[st][r * A_LD + c]), a[mi]);
        } else {
          const int k = ks + (lane & 7) + 8 * (lane >> 4), m = wm + mi * 16 + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(smem_u32(&As[st][k * AT_LD + m]), a[mi]);
        }
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int k = ks + (lane & 7) + 8 * ((lane >> 3) & 1), n = wn + np * 16 + 8 * (lane >> 4);
        ldsm_x4_t(smem_u32(&Bs[st][k * B_LD + n]), b[np]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const uint32_t* bb = b[ni >> 1];
          const int o = (ni & 1) * 2;
          mma_bf16_16816(acc[mi][ni], a[mi][0], a[mi][1], a[mi][2], a[mi][3], bb[o], bb[o + 1]);
        }
    }
    __syncthreads();    // this stage is refilled two iterations later
  }

  // epilogue: acc[mi][ni] = (m = g, n = 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
  const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = m0 + wm + mi * 16 + gq + 8 * h;
        const int n = n0 + wn + ni * 8 + 2 * t4;
        if (m >= mend || n >= g.N) continue;
        const float v0 = acc[mi][ni][2 * h], v1 = acc[mi][ni][2 * h + 1];
        const int64_t o = (int64_t)e * g.c_seg + (int64_t)m * g.ldc + n;
        if (EPI == GE_ACC_F32) {
          float2* p = reinterpret_cast<float2*>(reinterpret_cast<float*>(g.C) + o);
          float2 c = *p;
          c.x += v0;
          c.y += v1;
          *p = c;
        } else if (EPI == GE_STORE_F32) {
          *reinterpret_cast<float2*>(reinterpret_cast<float*>(g.C) + o) = make_float2(v0, v1);
        } else if (EPI == GE_STORE_BF16) {
          *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(g.C) + o) =
              (uint32_t)bf16_bits(v0) | ((uint32_t)bf16_bits(v1) << 16);
        } else {
          // GE_RELU2_GRAD: da = dh * 2 relu(a), with relu(a) = sqrt(h) from the
          // forward's stored h = relu(a)^2 (same [m][n] position in aux)
          const uint32_t hb = *reinterpret_cast<const uint32_t*>(g.aux + (int64_t)m * g.aux_ld + n);
          const float h0 = bf16_lo(hb), h1 = bf16_hi(hb);
          const float d0 = v0 * 2.f * sqrtf(h0), d1 = v1 * 2.f * sqrtf(h1);
          *reinterpret_cast<uint32_t*>(reinterpret_cast<bf16*>(g.C) + o) =
              (uint32_t)bf16_bits(d0) | ((uint32_t)bf16_bits(d1) << 16);
        }
      }
}

// 64-row tiles of the active segments: tprefix[j] = tiles of segments before
// active segment j, tprefix[n_active] = all (one CTA, n_active <= 1024)
__global__ void __launch_bounds__(1024) tile_scan_kernel(const int32_t* __restrict__ offsets,
                                                         const int32_t* __restrict__ active,
                                                         const WsHeader* __restrict__ hdr, int32_t* __restrict__ tprefix) {
  pdl_wait();
  __shared__ int wsum[32];
  const int na = hdr->n_active;
  const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
  int v = 0;
  if (j < na) {
    const int e = active[j];
    v = (offsets[e + 1] - offsets[e] + 63) / 64;
  }
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  if (j <= na) tprefix[j] = before + incl - v;    // j == na: v = 0, the total
}

// ---------------------------------------------------------------------------
// combine backward: packed row r = (t, k): dU[r] = bf16(w_tk dY[t]);
// q[t, k] = <dY[t], u[r]> / w_tk (u = w U is what the forward stored), FP32,
// summed by a fixed tree.  One CTA per packed row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_bwd_kernel(const bf16* __restrict__ dy, int64_t dy_ld,
                                                          const float* __restrict__ u, const int32_t* __restrict__ rt,
                                                          const int32_t* __restrict__ rs, const float* __restrict__ topw,
                                                          int K, int de, bf16* __restrict__ dU,
                                                          float* __restrict__ q) {
  pdl_wait();
  __shared__ float part[8];
  const int r = blockIdx.x;
  const int t = rt[r], k = rs[r];
  const float w = topw[(int64_t)t * K + k];
  const bf16* d = dy + (int64_t)t * dy_ld;
  const float* ur = u + (int64_t)r * de;
  float dot = 0.f;
  for (int c = threadIdx.x * 4; c < de; c += 256 * 4) {
    const uint2 db = *reinterpret_cast<const uint2*>(d + c);
    const float4 uv = *reinterpret_cast<const float4*>(ur + c);
    const float d0 = bf16_lo(db.x), d1 = bf16_hi(db.x), d2 = bf16_lo(db.y), d3 = bf16_hi(db.y);
    dot = fmaf(d0, uv.x, dot);
    dot = fmaf(d1, uv.y, dot);
    dot = fmaf(d2, uv.z, dot);
    dot = fmaf(d3, uv.w, dot);
    uint2 o;
    o.x = (uint32_t)bf16_bits(w * d0) | ((uint32_t)bf16_bits(w * d1) << 16);
    o.y = (uint32_t)bf16_bits(w * d2) | ((uint32_t)bf16_bits(w * d3) << 16);
    *reinterpret_cast<uint2*>(dU + (int64_t)r * de + c) = o;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = dot;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int i = 0; i < 8; ++i) s += part[i];
    q[(int64_t)t * K + k] = s / w;
  }
}

// gate backward of token t: the chosen scores s_k, S = sum_k s_k;
// ds_k = rsf / S (q_k - sum_j q_j s_j / S) (normalised) or rsf q_k;
// dz_k = ds_k s_k (1 - s_k).  One thread per token.
__global__ void gate_bwd_kernel(const float* __restrict__ scores, const int32_t* __restrict__ ids,
                                const float* __restrict__ q, int T, int E, int K, int norm, float rsf,
                                float* __restrict__ dz) {
  pdl_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  float S = 0.f, qs = 0.f;
  for (int k = 0; k < K; ++k) {
    const float s = scores[(int64_t)t * E + ids[(int64_t)t * K + k]];
    S += s;
    qs += q[(int64_t)t * K + k] * s;
  }
  for (int k = 0; k < K; ++k) {
    const float s = scores[(int64_t)t * E + ids[(int64_t)t * K + k]];
    const float qk = q[(int64_t)t * K + k];
    const float ds = norm ? rsf / S * (qk - qs / S) : rsf * qk;
    dz[(int64_t)t * K + k] = ds * s * (1.f - s);
  }
}

// router weight gradient: dW_r[e] += sum over expert e's packed rows r, in
// order, of dz[r] x[token r] (x: BF16 or FP32 rows).  Grid (d / 256, active).
template <bool XF32>
__global__ void router_wgrad_kernel(const void* __restrict__ x, int d, const float* __restrict__ dz,
                                    const int32_t* __restrict__ rt, const int32_t* __restrict__ rs, int K,
                                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ active,
                                    const WsHeader* __restrict__ hdr, float* __restrict__ dW) {
  pdl_wait();
  const int j = blockIdx.y;
  if (j >= hdr->n_active) return;
  const int e = active[j];
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= d) return;
  float acc = 0.f;
  for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
    const int t = rt[r];
    const float xv = XF32 ? reinterpret_cast<const float*>(x)[(int64_t)t * d + c]
                          : __bfloat162float(reinterpret_cast<const bf16*>(x)[(int64_t)t * d + c]);
    acc = fmaf(dz[(int64_t)t * K + rs[r]], xv, acc);
  }
  dW[(int64_t)e * d + c] += acc;
}

// dx[t] = (sum_k dz_tk W_r[id_tk]) + a[t] + b[t] (a, b: FP32 [T, d] or NULL),
// in that order.  Grid (d / 256, T).
__global__ void input_grad_kernel(const float* __restrict__ dz, const int32_t* __restrict__ ids, int K,
                                  const float* __restrict__ w_router, int d, const float* __restrict__ a,
                                  const float* __restrict__ b, float* __restrict__ dx) {
  pdl_wait();
  const int t = blockIdx.y;
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= d) return;
  float v = 0.f;
  for (int k = 0; k < K; ++k)
    v = fmaf(dz[(int64_t)t * K + k], w_router[(int64_t)ids[(int64_t)t * K + k] * d + c], v);
  if (a) v += a[(int64_t)t * d + c];
  if (b) v += b[(int64_t)t * d + c];
  dx[(int64_t)t * d + c] = v;
}

// RMSNorm backward of the block, one CTA per row: with r = 1 / sqrt(mean(x^2) + eps),
// dx = dout + r gamma dxn - r^3 x / d * sum_j gamma_j dxn_j x_j (written);
// xr = x * r per column is written to xr for the gamma gradient
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(const bf16* __restrict__ x, const float* __restrict__ gamma,
                                                          float eps, int d, const bf16* __restrict__ dout,
                                                          const float* __restrict__ dxn, float* __restrict__ dx,
                                                          float* __restrict__ xr) {
  pdl_wait();
  __shared__ float part[2][8];
  const int t = blockIdx.x;
  const bf16* xrow = x + (int64_t)t * d;
  const float* drow = dxn + (int64_t)t * d;
  float ss = 0.f, dot = 0.f;
  for (int c = threadIdx.x; c < d; c += 256) {
    const float xv = __bfloat162float(xrow[c]);
    ss = fmaf(xv, xv, ss);
    dot = fmaf(gamma[c] * drow[c], xv, dot);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, off);
    dot += __shfl_xor_sync(0xffffffffu, dot, off);
  }
  if ((threadIdx.x & 31) == 0) {
    part[0][threadIdx.x >> 5] = ss;
    part[1][threadIdx.x >> 5] = dot;
  }
  __syncthreads();
  float tss = 0.f, tdot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    tss += part[0][w];
    tdot += part[1][w];
  }
  const float r = 1.0f / sqrtf(tss / (float)d + eps);
  const float coef = r * r * r * tdot / (float)d;
  for (int c = threadIdx.x; c < d; c += 256) {
    const float xv = __bfloat162float(xrow[c]);
    dx[(int64_t)t * d + c] = __bfloat162float(dout[(int64_t)t * d + c]) + (r * gamma[c] * drow[c] - coef * xv);
    xr[(int64_t)t * d + c] = xv * r;
  }
}

// dgamma[c] += sum over rows t, in order, of dxn[t, c] xr[t, c]
__global__ void colsum_prod_kernel(const float* __restrict__ a, const float* __restrict__ b, int T, int d,
                                   float* __restrict__ out) {
  pdl_wait();
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= d) return;
  float acc = 0.f;
  for (int t = 0; t < T; ++t) acc = fmaf(a[(int64_t)t * d + c], b[(int64_t)t * d + c], acc);
  out[c] += acc;
}

}  // namespace

cudaError_t launch_tile_scan(const int32_t* offsets, const int32_t* active, const WsHeader* hdr, int32_t* tprefix,
                             cudaStream_t s) {
  launch_k(tile_scan_kernel, 1, 1024, 0, s, offsets, active, hdr, tprefix);
  return cudaGetLastError();
}

cudaError_t launch_gemm_bwd(const GemmArgs& g, int segs, int rows, cudaStream_t s) {
  if (segs <= 0) return cudaSuccess;
  if (g.N % 8 || (g.mode == GM_ROWS && g.K % BK) || (g.mode == GM_KSEG && g.M % 8)) return cudaErrorInvalidValue;
  dim3 grid;
  if (g.mode == GM_ROWS) {
    if (rows <= 0) return cudaSuccess;
    // grouped: at most ceil(rows / 64) + segs tiles (a partial tile a segment)
    const int64_t tiles = g.offsets ? ceil_div(rows, BM) + segs : ceil_div(rows, BM);
    if (g.offsets && !g.tprefix) return cudaErrorInvalidValue;
    grid = dim3((unsigned)ceil_div(g.N, BN), (unsigned)tiles, 1);
  } else {
    grid = dim3((unsigned)ceil_div(g.N, BN), (unsigned)ceil_div(g.M, BM), (unsigned)segs);
  }
  if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidValue;
#define MOE_G(AT, EP) launch_k(gemm_bwd_kernel<AT, EP>, grid, kGThreads, 0, s, g)
  switch (g.epi) {
    case GE_ACC_F32: if (g.a_t) MOE_G(true, GE_ACC_F32); else MOE_G(false, GE_ACC_F32); break;
    case GE_STORE_F32: if (g.a_t) MOE_G(true, GE_STORE_F32); else MOE_G(false, GE_STORE_F32); break;
    case GE_STORE_BF16: if (g.a_t) MOE_G(true, GE_STORE_BF16); else MOE_G(false, GE_STORE_BF16); break;
    default: if (g.a_t) MOE_G(true, GE_RELU2_GRAD); else MOE_G(false, GE_RELU2_GRAD); break;
  }
#undef MOE_G
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const void* dy, int64_t dy_ld, const float* u, const int32_t* rt, const int32_t* rs,
                               const float* topw, int R, int K, int de, void* dU, float* q, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  if (de % 4) return cudaErrorInvalidValue;
  launch_k(combine_bwd_kernel, (unsigned)R, 256, 0, s, reinterpret_cast<const bf16*>(dy), dy_ld, u, rt, rs, topw, K,
           de, reinterpret_cast<bf16*>(dU), q);
  return cudaGetLastError();
}

cudaError_t launch_gate_bwd(const float* scores, const int32_t* ids, const float* q, int T, int E, int K, int norm,
                            float rsf, float* dz, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  launch_k(gate_bwd_kernel, (unsigned)ceil_div(T, 128), 128, 0, s, scores, ids, q, T, E, K, norm, rsf, dz);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const void* x, bool x_f32, int d, const float* dz, const int32_t* rt,
                                const int32_t* rs, int K, const int32_t* offsets, const int32_t* active,
                                const WsHeader* hdr, int segs, float* dW, cudaStream_t s) {
  if (segs <= 0) return cudaSuccess;
  const dim3 grid((unsigned)ceil_div(d, 256), (unsigned)segs);
  if (x_f32)
    launch_k(router_wgrad_kernel<true>, grid, 256, 0, s, x, d, dz, rt, rs, K, offsets, active, hdr, dW);
  else
    launch_k(router_wgrad_kernel<false>, grid, 256, 0, s, x, d, dz, rt, rs, K, offsets, active, hdr, dW);
  return cudaGetLastError();
}

cudaError_t launch_input_grad(const float* dz, const int32_t* ids, int T, int K, const float* w_router, int d,
                              const float* a, const float* b, float* dx, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  launch_k(input_grad_kernel, dim3((unsigned)ceil_div(d, 256), (unsigned)T), 256, 0, s, dz, ids, K, w_router, d, a, b,
           dx);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bwd(const void* x, const float* gamma, float eps, int T, int d, const void* dout,
                               const float* dxn, float* dx, float* xr, float* dgamma, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  launch_k(rmsnorm_bwd_kernel, (unsigned)T, 256, 0, s, reinterpret_cast<const bf16*>(x), gamma, eps, d,
           reinterpret_cast<const bf16*>(dout), dxn, dx, xr);
  if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
  if (dgamma) launch_k(colsum_prod_kernel, (unsigned)ceil_div(d, 256), 256, 0, s, dxn, xr, T, d, dgamma);
  return cudaGetLastError();
}

}  // namespace moe
