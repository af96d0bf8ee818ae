// ReLU^2-sparse down projection for decode (page "Nemotron-3.5-Super 120B on
// an 8 GB GPU", section "The engine, step by step", item 4 "Skip the zeros":
// after ReLU^2 most of an expert's neurons are exactly zero for a token, a
// zero neuron needs no column of the down matrix, and since NVFP4 shares one
// scale per 16 consecutive values the down matrix is re-laid once so that
// whole 16-neuron groups can be skipped; section "What didn't work": skipping
// single neurons lost to re-reading scales, 16-neuron groups won).
//
// Group-major down weights.  For expert e, 16-neuron group g (neurons
// 16g .. 16g+15) and 16-output tile o (outputs 16o .. 16o+15) the 16 x 16
// block of W_down[e] is stored contiguously, in the order the m16n8k16 MMA
// fragments take it, so one 16-byte load per thread brings a warp its whole
// A operand.  Lane l = 4r + t (r = l / 4, t = l % 4) of a block holds
//   output 16o + r,     neurons 16g + 4t .. 16g + 4t + 3, then
//   output 16o + r + 8, neurons 16g + 4t .. 16g + 4t + 3,
// and the MMA k positions {2t, 2t+1, 2t+8, 2t+9} stand for neurons
// 4t .. 4t+3 (the activation operand takes the same neurons, so the product
// is unchanged).  Every block of group g lies in one range of de x 16 values:
//   BF16:  Wg[e][g][o][l][8]                     (bf16, 16 bytes a lane)
//   NVFP4: Vg[e][g][q][l][4 tiles][2 + 2 bytes]  (the E2M1 bytes of the two
//          rows above for the 4 tiles of a 64-output quad q; each byte keeps
//          its two neurons, low nibble = even neuron: a byte permutation)
//          Sg[e][g][q][r][4 tiles][2]            (E4M3 scales of outputs
//          64q + 16j + r and 64q + 16j + r + 8 for group g)
//
// The kernels find an expert's live groups (any row of the expert with a
// nonzero h value in the group) and stream only those groups' weights; dead
// groups add exact zeros in the dense product, so skipping them changes no
// term of the sum.  The live groups are summed in ascending order, split over
// the warps in a fixed pattern and reduced in warp order: the result does not
// depend on scheduling.
#include "epilogue.cuh"
#include "nvfp4.cuh"

#include <cuda_fp16.h>

namespace moe {

namespace {

constexpr int kSpWarps = 8;
constexpr int kSpThreads = kSpWarps * 32;
constexpr int kSpMaxGroups = 1024;       // I / 16
constexpr int kSpNT = 2;                 // 8-row column blocks per pass
constexpr int kSpU = 4;                  // groups in flight per warp

struct SpSeg {
  int id, row0, nrows;
};

__device__ __forceinline__ bool sp_segment(const GemvArgs& a, SpSeg& s) {
  const int j = blockIdx.y;
  const int n_active = a.hdr->n_active;
  const int id = a.active[j];
  if (j >= n_active) return false;
  s.id = id;
  s.row0 = a.offsets[id];
  s.nrows = a.offsets[id + 1] - s.row0;
  return s.nrows > 0;
}

// Ascending list of the groups of 16 h values that hold a nonzero in any of
// the segment's rows (h 16-bit: BF16 or FP16; a -0 counts as zero, anything
// else, NaN included, as live).  Returns the count; every thread sees it.
__device__ int sp_live_groups(const GemvArgs& a, const SpSeg& sg, int ngroups, int* list, int* wc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* h = reinterpret_cast<const uint16_t*>(a.X);
  int total = 0;
  for (int base = 0; base < ngroups; base += kSpThreads) {
    const int grp = base + threadIdx.x;
    bool live = false;
    if (grp < ngroups) {
      for (int r = 0; r < sg.nrows && !live; ++r) {
        const uint4* p = reinterpret_cast<const uint4*>(h + (int64_t)(sg.row0 + r) * a.x_ld + 16 * grp);
        const uint4 q0 = p[0], q1 = p[1];
        const uint32_t any = (q0.x | q0.y | q0.z | q0.w | q1.x | q1.y | q1.z | q1.w) & 0x7FFF7FFFu;
        live = any != 0;
      }
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, live);
    if (lane == 0) wc[warp] = __popc(bal);
    __syncthreads();
    int before = total;
    for (int w = 0; w < warp; ++w) before += wc[w];
    if (live) list[before + __popc(bal & ((1u << lane) - 1u))] = grp;
    for (int w = 0; w < kSpWarps; ++w) total += wc[w];
    __syncthreads();   // wc is rewritten by the next chunk
  }
  return total;
}

// BF16 weights and h.  A CTA owns FPC outputs (FPC / 16 tiles); the warps of a
// tile split the live groups; rows in passes of 16.
template <int FPC>
__global__ void __launch_bounds__(kSpThreads) sparse_down_bf16_kernel(const GemvArgs a) {
  pdl_wait();
  constexpr int TILES = FPC / 16;
  constexpr int WG = kSpWarps / TILES;
  __shared__ int list[kSpMaxGroups];
  __shared__ int wc[kSpWarps];
  __shared__ float red[kSpWarps][kSpNT][128];
  __shared__ float wrs[kSpNT * 8];
  SpSeg sg;
  if (!sp_segment(a, sg)) return;
  const int nlive = sp_live_groups(a, sg, a.K / 16, list, wc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int kw = warp % WG;
  const int ot = blockIdx.x * TILES + warp / WG;
  const int n_ot = a.N / 16;
  const uint4* Wt = reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(a.W) + (int64_t)sg.id * a.w_seg_stride) +
                    (int64_t)ot * 32 + lane;
  const int64_t gstride = (int64_t)n_ot * 32;     // uint4s between groups
  const bf16* H = reinterpret_cast<const bf16*>(a.X);

  for (int p0 = 0; p0 < sg.nrows; p0 += kSpNT * 8) {
    const int prow = min(sg.nrows - p0, kSpNT * 8);
    if (p0 > 0) __syncthreads();                   // the previous pass is done with red and wrs
    if (threadIdx.x < prow) wrs[threadIdx.x] = route_weight(a, sg.row0 + p0 + threadIdx.x);
    const bf16* xr[kSpNT];
    bool xv[kSpNT];
#pragma unroll
    for (int j = 0; j < kSpNT; ++j) {
      const int r = j * 8 + g;
      xv[j] = r < prow;
      xr[j] = H + (int64_t)(sg.row0 + p0 + (xv[j] ? r : 0)) * a.x_ld + 4 * t4;
    }
    float acc[kSpNT][4];
#pragma unroll
    for (int j = 0; j < kSpNT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    for (int i = kw; i < nlive; i += WG * kSpU) {
      uint4 A[kSpU];
      int gg[kSpU];
#pragma unroll
      for (int u = 0; u < kSpU; ++u) {
        const int ii = i + WG * u;
        gg[u] = ii < nlive ? list[ii] : -1;
        if (gg[u] >= 0) A[u] = ldg_stream(Wt + gg[u] * gstride);
      }
#pragma unroll
      for (int u = 0; u < kSpU; ++u) {
        if (gg[u] < 0) continue;
#pragma unroll
        for (int j = 0; j < kSpNT; ++j) {
          if (j * 8 < prow) {
            uint2 B = make_uint2(0u, 0u);
            if (xv[j]) B = *reinterpret_cast<const uint2*>(xr[j] + 16 * gg[u]);
            mma_bf16_16816(acc[j], A[u].x, A[u].z, A[u].y, A[u].w, B.x, B.y);
          }
        }
      }
    }
    // acc[j][0]: (output g, row 2t), [1]: (g, 2t+1), [2]: (g+8, 2t), [3]: (g+8, 2t+1)
#pragma unroll
    for (int j = 0; j < kSpNT; ++j) {
      red[warp][j][g * 8 + 2 * t4] = acc[j][0];
      red[warp][j][g * 8 + 2 * t4 + 1] = acc[j][1];
      red[warp][j][(g + 8) * 8 + 2 * t4] = acc[j][2];
      red[warp][j][(g + 8) * 8 + 2 * t4 + 1] = acc[j][3];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < TILES * kSpNT * 128; o += kSpThreads) {
      const int ti = o / (kSpNT * 128), j = (o >> 7) % kSpNT, idx = o & 127;
      const int f = idx >> 3, r = j * 8 + (idx & 7);
      if (r < prow) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < WG; ++w) v += red[ti * WG + w][j][idx];
        epilogue_pre<EPI_SCALE, true, false>(a, sg.row0 + p0 + r, (blockIdx.x * TILES + ti) * 16 + f, v, 1.f,
                                             wrs[r]);
      }
    }
  }
}

// NVFP4 weights, FP16 h (the layer's FP16 decode path).  A CTA owns one quad
// of 64 outputs (4 tiles); its 8 warps split the live groups; each thread's
// 16-byte load holds its A fragments of all 4 tiles, its 8-byte scale load
// the scales of its two rows in each tile.  E2M1 x E4M3 products are exact in
// FP16; the MMA accumulates in FP32 and the per-tensor scale multiplies the
// FP32 sum.
__global__ void __launch_bounds__(kSpThreads, 3) sparse_down_nvfp4_kernel(const GemvArgs a) {
  pdl_wait();
  __shared__ int list[kSpMaxGroups];
  __shared__ int wc[kSpWarps];
  __shared__ float red[kSpWarps][kSpNT][4 * 128];
  __shared__ float wrs[kSpNT * 8];
  SpSeg sg;
  if (!sp_segment(a, sg)) return;
  const float gs = a.W_gs[sg.id];
  const int nlive = sp_live_groups(a, sg, a.K / 16, list, wc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int q = blockIdx.x, n_q = a.N / 64;
  const uint4* V = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(a.W) + sg.id * a.w_seg_stride) +
                   (int64_t)q * 32 + lane;
  const uint2* S = reinterpret_cast<const uint2*>(a.W_sf + sg.id * a.sf_seg_stride) + (int64_t)q * 8 + g;
  const int64_t vstride = (int64_t)n_q * 32, sstride = (int64_t)n_q * 8;
  const __half* H = reinterpret_cast<const __half*>(a.X);

  for (int p0 = 0; p0 < sg.nrows; p0 += kSpNT * 8) {
    const int prow = min(sg.nrows - p0, kSpNT * 8);
    if (p0 > 0) __syncthreads();
    if (threadIdx.x < prow) wrs[threadIdx.x] = route_weight(a, sg.row0 + p0 + threadIdx.x);
    const __half* xr[kSpNT];
    bool xv[kSpNT];
#pragma unroll
    for (int j = 0; j < kSpNT; ++j) {
      const int r = j * 8 + g;
      xv[j] = r < prow;
      xr[j] = H + (int64_t)(sg.row0 + p0 + (xv[j] ? r : 0)) * a.x_ld + 4 * t4;
    }
    float acc[kSpNT][4][4];
#pragma unroll
    for (int j = 0; j < kSpNT; ++j)
#pragma unroll
      for (int ti = 0; ti < 4; ++ti) acc[j][ti][0] = acc[j][ti][1] = acc[j][ti][2] = acc[j][ti][3] = 0.f;
    for (int i = warp; i < nlive; i += kSpWarps * kSpU) {
      uint4 Vq[kSpU];
      uint2 Sq[kSpU];
      int gg[kSpU];
#pragma unroll
      for (int u = 0; u < kSpU; ++u) {
        const int ii = i + kSpWarps * u;
        gg[u] = ii < nlive ? list[ii] : -1;
        if (gg[u] >= 0) {
          Vq[u] = ldg_stream(V + gg[u] * vstride);
          Sq[u] = __ldg(S + gg[u] * sstride);
        }
      }
#pragma unroll
      for (int u = 0; u < kSpU; ++u) {
        if (gg[u] < 0) continue;
        uint2 B[kSpNT];
#pragma unroll
        for (int j = 0; j < kSpNT; ++j) {
          B[j] = make_uint2(0u, 0u);
          if (j * 8 < prow && xv[j]) B[j] = *reinterpret_cast<const uint2*>(xr[j] + 16 * gg[u]);
        }
        const uint32_t vw[4] = {Vq[u].x, Vq[u].y, Vq[u].z, Vq[u].w};
#pragma unroll
        for (int ti = 0; ti < 4; ++ti) {
          uint32_t p[4];                           // row r pairs (4t, 4t+1), (4t+2, 4t+3); row r+8 the same
          e2m1x8_to_f16x2(vw[ti], p);
          const uint32_t s16 = (ti < 2 ? Sq[u].x : Sq[u].y) >> (16 * (ti & 1));
          const uint32_t sc = e4m3x2_to_f16x2(s16 & 0xFFFFu);    // (row r, row r + 8)
          const uint32_t s_lo = __byte_perm(sc, 0, 0x1010), s_hi = __byte_perm(sc, 0, 0x3232);
          const uint32_t a0 = hmul2_f16(p[0], s_lo), a2 = hmul2_f16(p[1], s_lo);
          const uint32_t a1 = hmul2_f16(p[2], s_hi), a3 = hmul2_f16(p[3], s_hi);
#pragma unroll
          for (int j = 0; j < kSpNT; ++j)
            if (j * 8 < prow) mma_f16_16816(acc[j][ti], a0, a1, a2, a3, B[j].x, B[j].y);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kSpNT; ++j)
#pragma unroll
      for (int ti = 0; ti < 4; ++ti) {
        float* rr = red[warp][j] + ti * 128;
        rr[g * 8 + 2 * t4] = acc[j][ti][0];
        rr[g * 8 + 2 * t4 + 1] = acc[j][ti][1];
        rr[(g + 8) * 8 + 2 * t4] = acc[j][ti][2];
        rr[(g + 8) * 8 + 2 * t4 + 1] = acc[j][ti][3];
      }
    __syncthreads();
    for (int o = threadIdx.x; o < kSpNT * 4 * 128; o += kSpThreads) {
      const int j = o / 512, ti = (o >> 7) & 3, idx = o & 127;
      const int f = idx >> 3, r = j * 8 + (idx & 7);
      if (r < prow) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kSpWarps; ++w) v += red[w][j][ti * 128 + idx];
        epilogue_pre<EPI_SCALE, true, false>(a, sg.row0 + p0 + r, q * 64 + ti * 16 + f, v, gs, wrs[r]);
      }
    }
  }
}

// ---- one-time re-layout of W_down into the group-major form ----------------
// BF16: one thread per destination 16-byte lane chunk (8 values)
__global__ void layout_bf16_kernel(const bf16* __restrict__ w, int E, int de, int I, uint4* __restrict__ out) {
  const int n_ot = de / 16, ng = I / 16;
  const int64_t n = (int64_t)E * ng * n_ot * 32;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < n; c += (int64_t)gridDim.x * blockDim.x) {
    const int l = (int)(c % 32);
    int64_t rest = c / 32;
    const int ot = (int)(rest % n_ot);
    rest /= n_ot;
    const int g = (int)(rest % ng);
    const int e = (int)(rest / ng);
    const int r = l >> 2, t = l & 3;
    const bf16* src = w + (int64_t)e * de * I;
    const int k0 = 16 * g + 4 * t;
    const uint2 lo = *reinterpret_cast<const uint2*>(src + (int64_t)(16 * ot + r) * I + k0);
    const uint2 hi = *reinterpret_cast<const uint2*>(src + (int64_t)(16 * ot + r + 8) * I + k0);
    out[c] = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
}

// NVFP4 values: one thread per destination 16-byte lane chunk; scales: one
// thread per destination 8-byte row chunk
__global__ void layout_nvfp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int E, int de,
                                    int I, uint4* __restrict__ vout, uint2* __restrict__ sout) {
  const int n_q = de / 64, ng = I / 16;
  const int64_t nv = (int64_t)E * ng * n_q * 32, ns = (int64_t)E * ng * n_q * 8;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < nv + ns; c += (int64_t)gridDim.x * blockDim.x) {
    if (c < nv) {
      const int l = (int)(c % 32);
      int64_t rest = c / 32;
      const int qd = (int)(rest % n_q);
      rest /= n_q;
      const int g = (int)(rest % ng);
      const int e = (int)(rest / ng);
      const int r = l >> 2, t = l & 3;
      const uint8_t* src = q + (int64_t)e * de * (I / 2);
      uint32_t w[4];
#pragma unroll
      for (int ti = 0; ti < 4; ++ti) {
        const int o = 64 * qd + 16 * ti + r;
        // neurons 16g + 4t .. +3 are bytes 8g + 2t, 8g + 2t + 1 of a row
        const uint16_t lo = *reinterpret_cast<const uint16_t*>(src + (int64_t)o * (I / 2) + 8 * g + 2 * t);
        const uint16_t hi = *reinterpret_cast<const uint16_t*>(src + (int64_t)(o + 8) * (I / 2) + 8 * g + 2 * t);
        w[ti] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      vout[c] = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      const int64_t cs = c - nv;
      const int r = (int)(cs % 8);
      int64_t rest = cs / 8;
      const int qd = (int)(rest % n_q);
      rest /= n_q;
      const int g = (int)(rest % ng);
      const int e = (int)(rest / ng);
      const uint8_t* src = sf + (int64_t)e * de * (I / 16);
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int ti = 0; ti < 4; ++ti) {
        const int o = 64 * qd + 16 * ti + r;
        const uint32_t b0 = src[(int64_t)o * (I / 16) + g], b1 = src[(int64_t)(o + 8) * (I / 16) + g];
        w[ti >> 1] |= (b0 | (b1 << 8)) << (16 * (ti & 1));
      }
      sout[cs] = make_uint2(w[0], w[1]);
    }
  }
}

}  // namespace

bool sparse_down_fits(int N, int K, bool nvfp4) {
  if (K % 16 || K / 16 > kSpMaxGroups) return false;
  return nvfp4 ? N % 64 == 0 : N % 32 == 0;
}

cudaError_t launch_sparse_down(const GemvArgs& a, bool nvfp4, int segs, cudaStream_t s) {
  if (segs <= 0) return cudaSuccess;
  if (!sparse_down_fits(a.N, a.K, nvfp4) || !a.offsets || !a.active || !a.hdr) return cudaErrorInvalidValue;
  if (nvfp4) {
    launch_k(sparse_down_nvfp4_kernel, dim3((unsigned)(a.N / 64), segs, 1), kSpThreads, 0, s, a);
  } else {
    launch_k(sparse_down_bf16_kernel<32>, dim3((unsigned)(a.N / 32), segs, 1), kSpThreads, 0, s, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_sparse_down_layout(const void* w, const uint8_t* sf, int E, int de, int I, bool nvfp4, void* out,
                                      void* out_sf, cudaStream_t s) {
  if (!sparse_down_fits(de, I, nvfp4)) return cudaErrorInvalidValue;
  const unsigned grid = 152 * 8;
  if (nvfp4)
    launch_k(layout_nvfp4_kernel, grid, 256, 0, s, reinterpret_cast<const uint8_t*>(w), sf, E, de, I,
             reinterpret_cast<uint4*>(out), reinterpret_cast<uint2*>(out_sf));
  else
    launch_k(layout_bf16_kernel, grid, 256, 0, s, reinterpret_cast<const bf16*>(w), E, de, I,
             reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace moe
