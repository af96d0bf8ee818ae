// Dispatch: per-expert route counts, exclusive scan, and the stable
// expert-contiguous layout of routes sorted by (expert, token, slot)
// (page "M6.1 - Routed Capacity: MoE Experts, Routers, and Token Dispatch",
// section 0x05A "The Route Row Is The Reversible Unit": offsets are the
// prefix sum of counts; section 0x05B: X_packed[j] = H[a_pi(j)]).
//
// Atomic-free: a warp walks a contiguous range of routes 32 at a time; lanes
// holding the same expert find each other with __match_any_sync, the lowest
// such lane adds the group size to the warp's private histogram row, and a
// lane's rank inside its group is the popcount of lower peers.  Per-expert
// bases are exclusive scans over (tile, warp) in index order, so route r lands
// after every earlier route of the same expert: the order is (expert, r) =
// (expert, token, slot) because a token names an expert at most once.
#include "nvfp4.cuh"
#include "select.cuh"

#include <algorithm>

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = 32;
constexpr int kTileTokens = 256;   // tokens per CTA in the multi-CTA path

// exclusive scan of one int per thread over a 1024-thread block
__device__ int block_exclusive_scan(int v, int* tmp32, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) tmp32[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = tmp32[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    tmp32[lane] = w;  // inclusive
  }
  __syncthreads();
  const int base = warp ? tmp32[warp - 1] : 0;
  if (total) *total = tmp32[31];
  __syncthreads();
  return base + x - v;
}

// Histogram of routes [r0, r1) into hist[warp][E] (warp-private rows).
__device__ void warp_histograms(const int32_t* __restrict__ ids, int r0, int r1, int E, int* hist,
                                int32_t* err) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = r1 - r0;
  const int per = (int)ceil_div(ceil_div(n, kWarps), 32) * 32;
  const int b = r0 + warp * per, bend = min(r1, b + per);
  for (int base = b; base < bend; base += 32) {
    const int r = base + lane;
    int e = -1;
    if (r < bend) {
      e = ids[r];
      if (e < 0 || e >= E) { set_error(err, MOE_DEVERR_EXPERT_ID); e = -1; }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

// Scatter of routes [r0, r1) using per-warp running bases hist[warp][E].
__device__ void warp_scatter(const int32_t* __restrict__ ids, int r0, int r1, int E, int K, int* hist,
                             int32_t* route_token, int32_t* route_slot, int32_t* token_slot_row) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = r1 - r0;
  const int per = (int)ceil_div(ceil_div(n, kWarps), 32) * 32;
  const int b = r0 + warp * per, bend = min(r1, b + per);
  for (int base = b; base < bend; base += 32) {
    const int r = base + lane;
    int e = -1;
    if (r < bend) {
      e = ids[r];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int pos = -1;
    if (e >= 0) pos = hist[warp * E + e] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) hist[warp * E + e] += __popc(peers);
    __syncwarp();
    if (r < bend) {
      token_slot_row[r] = pos;
      if (pos >= 0) {
        route_token[pos] = r / K;
        route_slot[pos] = r % K;
      }
    }
  }
}

// x_packed[j] = x_e[route_token[j]]: one warp per packed row, every 16-byte
// piece of the row loaded before any is stored.  TO_F16: BF16 rows are stored
// as their FP16 copies (exact inside FP16's range).
template <bool TO_F16>
__global__ void __launch_bounds__(256) pack_rows_kernel(const uint4* __restrict__ x_e,
                                                        const int32_t* __restrict__ route_token,
                                                        const int32_t* __restrict__ offsets, int E, int row_vecs,
                                                        uint4* __restrict__ x_packed, int32_t* __restrict__ err) {
  pdl_wait();
  const int R = offsets[E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = blockIdx.x * 8 + warp; j < R; j += gridDim.x * 8) {
    const uint4* src = x_e + (int64_t)route_token[j] * row_vecs;
    uint4* dst = x_packed + (int64_t)j * row_vecs;
    constexpr int U = 6;
    for (int v0 = lane; v0 < row_vecs; v0 += 32 * U) {
      uint4 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (v0 + 32 * u < row_vecs) q[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (v0 + 32 * u >= row_vecs) continue;
        if (TO_F16) {
          if (err && bf16x4_beyond_f16(q[u])) set_error(err, MOE_DEVERR_RANGE);
          q[u] = make_uint4(bf16x2_to_f16x2(q[u].x), bf16x2_to_f16x2(q[u].y), bf16x2_to_f16x2(q[u].z),
                            bf16x2_to_f16x2(q[u].w));
        }
        dst[v0 + 32 * u] = q[u];
      }
    }
  }
}

// Experts with routes, in ascending id, and the tensor-core tile prefix.
__device__ void write_schedule(const DispatchArgs& a, int e, int total, int off, int* tmp32) {
  const int has = (e < a.E && total > 0) ? 1 : 0;
  int n_active = 0;
  const int pos = block_exclusive_scan(has, tmp32, &n_active);
  if (has) a.active[pos] = e;
  int tiles = 0;
  if (a.tile_rows > 0 && e < a.E) tiles = (int)ceil_div(total, a.tile_rows);
  int n_tiles = 0;
  const int tpos = block_exclusive_scan(tiles, tmp32, &n_tiles);
  if (a.tile_prefix && e < a.E) a.tile_prefix[e] = tpos;
  if (a.tile_prefix && e == a.E - 1) a.tile_prefix[a.E] = tpos + tiles;
  // largest count: reduce via shuffles + shared
  int m = (e < a.E) ? total : 0;
#pragma unroll
  for (int off2 = 16; off2 > 0; off2 >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off2));
  if ((threadIdx.x & 31) == 0) tmp32[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    int mm = 0;
    for (int w = 0; w < kWarps; ++w) mm = max(mm, tmp32[w]);
    a.hdr->n_active = n_active;
    a.hdr->n_tiles = n_tiles;
    a.hdr->max_rows = mm;
  }
  if (e < a.E) {
    a.counts[e] = total;
    a.offsets[e] = off;
    if (e == a.E - 1) a.offsets[a.E] = off + total;
  }
}

// ---------------------------------------------------------------------------
// single CTA (few routes)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) dispatch_single(const DispatchArgs a) {
  pdl_wait();
  extern __shared__ int sm[];
  int* hist = sm;                      // [32][E]
  int* tmp32 = sm + kWarps * a.E;      // [32]
  const int R = a.T * a.K;
  for (int i = threadIdx.x; i < kWarps * a.E; i += kThreads) hist[i] = 0;
  __syncthreads();
  warp_histograms(a.ids, 0, R, a.E, hist, &a.hdr->err);
  __syncthreads();
  const int e = threadIdx.x;
  int total = 0;
  if (e < a.E) {
    for (int w = 0; w < kWarps; ++w) {
      const int c = hist[w * a.E + e];
      hist[w * a.E + e] = total;
      total += c;
    }
  }
  const int off = block_exclusive_scan(e < a.E ? total : 0, tmp32, nullptr);
  if (e < a.E)
    for (int w = 0; w < kWarps; ++w) hist[w * a.E + e] += off;
  write_schedule(a, e, total, off, tmp32);
  __syncthreads();
  warp_scatter(a.ids, 0, R, a.E, a.K, hist, a.route_token, a.route_slot, a.token_slot_row);
}

// ---------------------------------------------------------------------------
// multi CTA (many routes): count per token tile, one scan CTA, scatter
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) dispatch_count(const DispatchArgs a) {
  pdl_wait();
  extern __shared__ int sm[];
  int* hist = sm;
  const int tile = blockIdx.x;
  const int r0 = tile * kTileTokens * a.K;
  const int r1 = min(a.T, (tile + 1) * kTileTokens) * a.K;
  for (int i = threadIdx.x; i < kWarps * a.E; i += kThreads) hist[i] = 0;
  __syncthreads();
  warp_histograms(a.ids, r0, r1, a.E, hist, &a.hdr->err);
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += kThreads) {
    int s = 0;
    for (int w = 0; w < kWarps; ++w) s += hist[w * a.E + e];
    a.tile_counts[(int64_t)tile * a.E + e] = s;
  }
}

__global__ void __launch_bounds__(kThreads) dispatch_scan(const DispatchArgs a, int n_tiles) {
  pdl_wait();
  __shared__ int tmp32[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < a.E) {
    for (int tl = 0; tl < n_tiles; ++tl) {
      const int c = a.tile_counts[(int64_t)tl * a.E + e];
      a.tile_counts[(int64_t)tl * a.E + e] = total;
      total += c;
    }
  }
  const int off = block_exclusive_scan(e < a.E ? total : 0, tmp32, nullptr);
  if (e < a.E)
    for (int tl = 0; tl < n_tiles; ++tl) a.tile_counts[(int64_t)tl * a.E + e] += off;
  write_schedule(a, e, total, off, tmp32);
}

__global__ void __launch_bounds__(kThreads) dispatch_scatter(const DispatchArgs a) {
  pdl_wait();
  extern __shared__ int sm[];
  int* hist = sm;
  const int tile = blockIdx.x;
  const int r0 = tile * kTileTokens * a.K;
  const int r1 = min(a.T, (tile + 1) * kTileTokens) * a.K;
  for (int i = threadIdx.x; i < kWarps * a.E; i += kThreads) hist[i] = 0;
  __syncthreads();
  warp_histograms(a.ids, r0, r1, a.E, hist, nullptr);
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += kThreads) {
    int run = a.tile_counts[(int64_t)tile * a.E + e];
    for (int w = 0; w < kWarps; ++w) {
      const int c = hist[w * a.E + e];
      hist[w * a.E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  warp_scatter(a.ids, r0, r1, a.E, a.K, hist, a.route_token, a.route_slot, a.token_slot_row);
}

// ---------------------------------------------------------------------------
// a few tokens (T <= 16, T*K <= 256): selection and dispatch in one CTA.  Warp t
// selects token t (the selection kernel's code), then every route r is placed
// directly: its packed position is the number of routes ordered before it by
// (expert, r); an expert's offset is the number of routes with a lower expert.
// Same outputs as the selection kernel followed by dispatch_single.
// ---------------------------------------------------------------------------
constexpr int kTinyThreads = 512;
constexpr int kTinyMaxRoutes = 256;   // the placement below is quadratic in the routes
constexpr int kTinyMaxTokens = kTinyThreads / 32;

template <int P>
__global__ void __launch_bounds__(kTinyThreads) select_dispatch_tiny(const SelectArgs sa, const DispatchArgs a) {
  pdl_wait();
  __shared__ int sid[kTinyMaxRoutes];     // expert of route r (-1: invalid)
  __shared__ int first[kTinyMaxRoutes];   // route r is its expert's first route
  __shared__ int cnt_max[kTinyThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (a.T == 1 && sa.E >= 256 && cta_select_fits(kTinyThreads, sa.E, sa.G, sa.TG, sa.K))
    // one token of a wide router: all 16 warps select it, an expert a thread
    // (Super latent layer at one token 0.094 -> 0.090 ms, Super NVFP4 0.0794 ->
    // 0.0779; for the 128-expert router one warp measured faster, 0.0502 vs
    // 0.0518 ms)
    select_token_cta<kTinyThreads>(sa.logits, sa.nparts, sa.part_stride, sa.logits_out, 0, sa.E, sa.bias, sa.G,
                                   sa.TG, sa.K, sa.norm, sa.rsf, sa.scores, sa.ids, sa.w, sa.err);
  else if (warp < a.T)
    select_token<P>(sa.logits, sa.nparts, sa.part_stride, sa.logits_out, warp, sa.E, sa.bias, sa.G, sa.TG, sa.K,
                    sa.norm, sa.rsf, sa.scores, sa.ids, sa.w, sa.err, warp, lane, a.T > 8);
  __syncthreads();                        // this CTA's id writes are visible to it
  const int R = a.T * a.K;
  const int r = threadIdx.x;
  int e = -1;
  if (r < R) {
    e = a.ids[r];
    if (e < 0 || e >= a.E) {
      set_error(&a.hdr->err, MOE_DEVERR_EXPERT_ID);
      e = -1;
    }
    sid[r] = e;
  }
  __syncthreads();
  if (r < R) {
    int pos = -1;
    bool is_first = e >= 0;
    if (e >= 0) {
      pos = 0;
      for (int j = 0; j < R; ++j) {
        const int ej = sid[j];
        pos += (ej >= 0) && (ej < e || (ej == e && j < r));
        is_first &= !(ej == e && j < r);
      }
    }
    first[r] = is_first ? 1 : 0;
    a.token_slot_row[r] = pos;
    if (pos >= 0) {
      a.route_token[pos] = r / a.K;
      a.route_slot[pos] = r % a.K;
    }
  }
  __syncthreads();
  // per expert: count, offset; the active list (experts with routes, ascending)
  int local_max = 0;
  for (int x = threadIdx.x; x <= a.E; x += kTinyThreads) {
    int below = 0, count = 0;
    for (int j = 0; j < R; ++j) {
      const int ej = sid[j];
      below += (ej >= 0 && ej < x);
      count += (ej == x);
    }
    a.offsets[x] = below;
    if (x < a.E) {
      a.counts[x] = count;
      local_max = max(local_max, count);
    }
  }
  if (r < R && first[r]) {
    int idx = 0;                          // distinct experts below this one
    for (int j = 0; j < R; ++j) idx += first[j] && sid[j] < e;
    a.active[idx] = e;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) local_max = max(local_max, __shfl_xor_sync(0xffffffffu, local_max, off));
  if (lane == 0) cnt_max[warp] = local_max;
  __syncthreads();
  if (threadIdx.x == 0) {
    int n_active = 0, mm = 0;
    for (int j = 0; j < R; ++j) n_active += first[j];
    for (int w = 0; w < kTinyThreads / 32; ++w) mm = max(mm, cnt_max[w]);
    a.hdr->n_active = n_active;
    a.hdr->n_tiles = 0;
    a.hdr->max_rows = mm;
  }
}

constexpr int kSingleMaxRoutes = 4096;

// the dynamic shared-memory limits are raised once per device, to the largest expert count
PerDeviceOnce g_attr_single, g_attr_multi;

cudaError_t launch_pack(const DispatchArgs& a, cudaStream_t s) {
  if (!a.x_packed || !a.x_e) return cudaSuccess;
  return launch_pack_rows(a.x_e, a.route_token, a.offsets, a.E, a.T * a.K, a.de, a.elem_bytes, a.pack_f16,
                          a.x_packed, s, &a.hdr->err);
}

}  // namespace

cudaError_t launch_pack_rows(const void* x_e, const int32_t* route_token, const int32_t* offsets, int E, int R,
                             int de, int elem_bytes, bool to_f16, void* x_packed, cudaStream_t s, int32_t* err) {
  if (R <= 0) return cudaSuccess;
  if ((to_f16 && elem_bytes != 2) || (de * elem_bytes) % 16) return cudaErrorNotSupported;
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(R, 8), 16384);
  launch_k(to_f16 ? pack_rows_kernel<true> : pack_rows_kernel<false>, grid, 256, 0, s,
           reinterpret_cast<const uint4*>(x_e), route_token, offsets, E, de * elem_bytes / 16,
           reinterpret_cast<uint4*>(x_packed), err);
  return cudaGetLastError();
}

bool select_dispatch_fits(int T, int K, const DispatchArgs& a) {
  return T >= 1 && T <= kTinyMaxTokens && T * K <= kTinyMaxRoutes && a.tile_rows == 0 && !a.x_packed;
}

cudaError_t launch_select_dispatch(const SelectArgs& sa, const DispatchArgs& a, cudaStream_t s) {
  if (!select_dispatch_fits(a.T, a.K, a)) return cudaErrorNotSupported;
  const int P = (int)ceil_div(sa.E, 32);
#define MOE_TINY(PP) \
  launch_k(select_dispatch_tiny<PP>, 1, kTinyThreads, 0, s, sa, a); \
  return cudaGetLastError()
  if (P <= 1) { MOE_TINY(1); }
  if (P <= 2) { MOE_TINY(2); }
  if (P <= 4) { MOE_TINY(4); }
  if (P <= 8) { MOE_TINY(8); }
  if (P <= 16) { MOE_TINY(16); }
  MOE_TINY(32);
#undef MOE_TINY
}

size_t dispatch_tile_count_elems(int T, int K, int E) {
  (void)K;
  return (size_t)ceil_div(T, kTileTokens) * (size_t)E;
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
  const int R = a.T * a.K;
  if (R <= 0) return cudaSuccess;
  if (R <= kSingleMaxRoutes) {
    const size_t smem = (size_t)(kWarps * a.E + 32) * sizeof(int);
    cudaError_t e = g_attr_single.run([](int&) {
      return cudaFuncSetAttribute(dispatch_single, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)((kWarps * 1024 + 32) * sizeof(int)));
    });
    if (e != cudaSuccess) return e;
    launch_k(dispatch_single, 1, kThreads, smem, s, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pack(a, s);
  }
  const int n_tiles = (int)ceil_div(a.T, kTileTokens);
  const size_t smem = (size_t)(kWarps * a.E) * sizeof(int);
  cudaError_t e = g_attr_multi.run([](int&) {
    const int most = (int)(kWarps * 1024 * sizeof(int));
    const cudaError_t r = cudaFuncSetAttribute(dispatch_count, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(dispatch_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
  });
  if (e != cudaSuccess) return e;
  launch_k(dispatch_count, n_tiles, kThreads, smem, s, a);
  launch_k(dispatch_scan, 1, kThreads, 0, s, a, n_tiles);
  launch_k(dispatch_scatter, n_tiles, kThreads, smem, s, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_pack(a, s);
}

}  // namespace moe
