// C ABI of the routed ReLU^2 MoE layer: argument checks, workspace layout and
// the order of the steps.  Every kernel launch goes to the caller's stream.
#include "internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

using namespace moe;

namespace moe {
static std::atomic<int64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace moe

namespace {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxGroups = 32;
constexpr int64_t kMaxRoutes = (int64_t)1 << 28;

constexpr int kDecodeMaxT = 64;   // up to this many tokens: weight-streaming GEMV; above: tensor cores

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// NVFP4 expert products: activation terms on the FP4 tensor path (1..4), 0
// for the FP16 path (weights decoded to FP16 inside the kernels), or -1 for
// the measured choice: kActTerms terms on the FP4 path from 8 to 64 tokens
// (a grouped decode product there streams the weights at 70-85 % of HBM
// against 45 % for the FP16 GEMV), the FP16 path below 8 tokens (where the
// GEMV's shorter launch chain wins: Super NVFP4 layer 0.081 vs 0.090 ms at 1
// token, 0.109 vs 0.115 ms at 4, equal at 8, 0.181 vs 0.207 ms at 16) and
// above 64 tokens (where quantising every routed row and h into terms costs
// more than the FP4 products save)
std::atomic<int> g_act_terms{-1};
constexpr int kFp4MinT = 8, kFp4MaxT = 64;

// activation terms a layer of T tokens uses on the FP4 path (0: FP16 path)
inline int act_terms_for(int T) {
  const int n = g_act_terms.load();
  if (n >= 0) return n;
  return T >= kFp4MinT && T <= kFp4MaxT ? kActTerms : 0;
}
inline int act_bytes(const moe_config_t* c) { return c->act_dtype == MOE_DT_F32 ? 4 : 2; }
inline int de_of(const moe_config_t* c) { return c->d_latent > 0 ? c->d_latent : c->d_model; }

struct Layout {
  size_t hdr, logits, logit_parts, scores, ids, topw, counts, offsets, active, tile_prefix, w_split;
  size_t route_token, route_slot, tsr, x_l, x_packed, h, u, y_r, y_rl, hs, ys, tile_counts;
  // NVFP4 experts: activation terms of the expert input rows and of h, their
  // block scales and row scales (sized for kActTermsMax terms)
  size_t xq, xq_sf, xq_g, hq, hq_sf, hq_g;
  size_t xn;   // the block's RMSNorm output rows [T, d] (activation type)
  size_t total;
};

inline size_t take(size_t& off, size_t bytes) {
  off = (off + 255) & ~(size_t)255;
  const size_t o = off;
  off += bytes;
  return o;
}

Layout make_layout(const moe_config_t* c, int32_t T) {
  Layout L{};
  const size_t t = (size_t)T, E = c->n_experts, K = c->top_k, R = t * K;
  const size_t de = de_of(c), ab = act_bytes(c);
  size_t off = 0;
  L.hdr = take(off, sizeof(WsHeader));
  L.logits = take(off, t * E * 4);
  L.logit_parts = take(off, T > 64 ? (size_t)kRouterParts * t * E * 4 : 0);   // K-split router logits
  L.scores = take(off, t * E * 4);
  L.ids = take(off, R * 4);
  L.topw = take(off, R * 4);
  L.counts = take(off, E * 4);
  L.offsets = take(off, (E + 1) * 4);
  L.active = take(off, E * 4);
  L.tile_prefix = take(off, (E + 1) * 4);
  L.w_split = take(off, E * 3 * (size_t)c->d_model * 2);
  L.route_token = take(off, R * 4);
  L.route_slot = take(off, R * 4);
  L.tsr = take(off, R * 4);
  L.x_l = take(off, c->d_latent > 0 ? t * c->d_latent * ab : 0);
  L.x_packed = take(off, R * de * ab);
  L.h = take(off, R * (size_t)c->d_expert * ab);
  L.u = take(off, R * de * 4);
  L.y_r = take(off, t * de * 4);
  L.y_rl = take(off, c->d_latent > 0 ? t * de * ab : 0);
  L.hs = take(off, t * (size_t)c->d_shared * ab);
  L.ys = take(off, t * (size_t)c->d_model * 4);
  L.tile_counts = take(off, dispatch_tile_count_elems(T, c->top_k, c->n_experts) * 4);
  const bool fp4 = c->expert_dtype == MOE_DT_NVFP4;
  const size_t nt = fp4 ? kActTermsMax : 0, I = c->d_expert;
  L.xq = take(off, nt * R * de / 2);
  L.xq_sf = take(off, nt * R * (size_t)act_sf_ld((int)de));
  L.xq_g = take(off, fp4 ? R * 4 : 0);
  L.hq = take(off, nt * R * I / 2);
  L.hq_sf = take(off, nt * R * (size_t)act_sf_ld((int)I));
  L.hq_g = take(off, fp4 ? R * 4 : 0);
  L.xn = take(off, t * (size_t)c->d_model * ab);
  L.total = (off + 255) & ~(size_t)255;
  return L;
}

moe_status_t check_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const int E = c->n_experts, K = c->top_k, G = c->n_group, TG = c->topk_group;
  if (c->d_model <= 0 || c->d_expert <= 0 || c->d_latent < 0 || c->d_shared < 0) return MOE_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (K < 1 || K > E || K > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (G < 1 || G > kMaxGroups || E % G != 0 || TG < 1 || TG > G) return MOE_ERR_INVALID_ARG;
  if (G > 1 && E / G < 2) return MOE_ERR_INVALID_ARG;          // a group score needs two members
  if ((int64_t)K > (int64_t)TG * (E / G)) return MOE_ERR_INVALID_ARG;
  if (c->norm_topk_prob != 0 && c->norm_topk_prob != 1) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->routed_scaling_factor)) return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_DT_F32 && c->act_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (c->expert_dtype != MOE_DT_F32 && c->expert_dtype != MOE_DT_BF16 && c->expert_dtype != MOE_DT_NVFP4)
    return MOE_ERR_INVALID_ARG;
  if ((c->expert_dtype == MOE_DT_F32) != (c->act_dtype == MOE_DT_F32)) return MOE_ERR_UNSUPPORTED;
  if (c->d_model % 64 || c->d_expert % 64 || c->d_latent % 64 || c->d_shared % 64) return MOE_ERR_UNSUPPORTED;
  if (c->expert_dtype == MOE_DT_NVFP4 && (de_of(c) % 128 || c->d_expert % 128)) return MOE_ERR_UNSUPPORTED;
  if (c->expert_dtype == MOE_DT_NVFP4 && c->act_dtype != MOE_DT_BF16) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_common(const moe_config_t* c, int32_t T, const void* ws, size_t ws_bytes) {
  moe_status_t st = check_config(c);
  if (st != MOE_OK) return st;
  if (T < 0 || (int64_t)T * c->top_k > kMaxRoutes) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < make_layout(c, T).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

#define REQ(p) do { if (!(p) || !aligned16(p)) return MOE_ERR_INVALID_ARG; } while (0)
#define OPT(p) do { if ((p) && !aligned16(p)) return MOE_ERR_INVALID_ARG; } while (0)
#define CU(x) do { if ((x) != cudaSuccess) return MOE_ERR_CUDA; } while (0)

inline int wfmt_of(const moe_config_t* c) {
  return c->expert_dtype == MOE_DT_F32 ? WF_F32 : (c->expert_dtype == MOE_DT_NVFP4 ? WF_NVFP4 : WF_BF16);
}
inline int dense_fmt(const moe_config_t* c) { return c->act_dtype == MOE_DT_F32 ? WF_F32 : WF_BF16; }

// tensor-core path: BF16 layers with more than kDecodeMaxT tokens
inline bool use_tc(const moe_config_t* c, int T) {
  return c->act_dtype == MOE_DT_BF16 && c->expert_dtype != MOE_DT_F32 && T > kDecodeMaxT;
}

inline bool fp4_path(const moe_config_t* c, int T);

// Dense products (shared expert, latent pair) run on the tensor cores above
// 64 tokens, and from 32 tokens when the expert products themselves run on
// the persistent FP4 kernels: at 32-64 rows the GEMV's 16-row passes are
// issue-bound (a 44 MB Super shared product took 46 us), and with the expert
// products on persistent kernels nothing overlaps them anyway (Super NVFP4
// layer at 64 tokens 0.329 -> 0.293 ms).  Next to streaming expert GEMVs the
// GEMV shared expert overlaps them and stays (Super BF16 at 64 tokens:
// 0.877 ms with GEMVs, 1.034 ms with tensor-core dense products).
constexpr int kDenseTcMinT = 32;
inline bool dense_tc(const moe_config_t* c, int T) {
  if (c->act_dtype != MOE_DT_BF16 || c->expert_dtype == MOE_DT_F32) return false;
  return T > kDecodeMaxT || (T >= kDenseTcMinT && fp4_path(c, T));
}

// dense product out[T, N] = X[T, K] W[N, K]^T through the GEMV or the tensor cores
cudaError_t run_dense(const moe_config_t* c, const GemvArgs& a, int epi, bool out_f32, int T, cudaStream_t s) {
  if (dense_tc(c, T))
    return launch_gemm_tc(a, epi, out_f32, a.N, T, 0, tc_tile_rows(T, 1, a.N), s);
  return launch_gemv(a, dense_fmt(c), c->act_dtype, epi, out_f32, T, 1, s);
}

GemvArgs dense_args(const void* W, int N, int K, const void* X, int rows, void* out, int64_t out_ld) {
  GemvArgs a{};
  a.W = W; a.N = N; a.K = K; a.X = X; a.x_ld = K; a.dense_rows = rows;
  a.out = out; a.out_ld = out_ld;
  return a;
}

struct Ptrs {
  char* base;
  Layout L;
  template <class T> T* at(size_t o) const { return reinterpret_cast<T*>(base + o); }
  WsHeader* hdr() const { return at<WsHeader>(L.hdr); }
};

// ---- steps -----------------------------------------------------------------
// router logits; the selection's arguments (the logits may be split over K parts)
moe_status_t run_logits(const moe_config_t* c, int T, const void* x, const float* w_router, const float* bias,
                        float* logits, float* scores, int32_t* ids, float* w, const Ptrs& P, cudaStream_t s,
                        SelectArgs& sa) {
  float* parts = T > 64 ? P.at<float>(P.L.logit_parts) : nullptr;
  int nparts = 1;
  CU(launch_router_logits(x, c->act_dtype, T, c->d_model, w_router, c->n_experts, logits, s,
                          P.at<void>(P.L.w_split), parts, &nparts));
  const bool split = nparts > 1;
  sa = SelectArgs{split ? parts : logits, nparts, (int64_t)T * c->n_experts, split ? logits : nullptr, T,
                  c->n_experts, bias, c->n_group, c->topk_group, c->top_k, c->norm_topk_prob,
                  c->routed_scaling_factor, scores, ids, w, &P.hdr()->err};
  return MOE_OK;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  return launch_router_select(a.logits, a.nparts, a.part_stride, a.logits_out, a.T, a.E, a.bias, a.G, a.TG, a.K,
                              a.norm, a.rsf, a.scores, a.ids, a.w, a.err, s);
}

moe_status_t run_router(const moe_config_t* c, int T, const void* x, const float* w_router, const float* bias,
                        float* logits, float* scores, int32_t* ids, float* w, const Ptrs& P, cudaStream_t s) {
  SelectArgs sa;
  moe_status_t st = run_logits(c, T, x, w_router, bias, logits, scores, ids, w, P, s, sa);
  if (st != MOE_OK) return st;
  CU(launch_select(sa, s));
  return MOE_OK;
}

DispatchArgs dispatch_args(const moe_config_t* c, int T, const int32_t* ids, const void* x_e, int32_t* counts,
                           int32_t* offsets, int32_t* rt, int32_t* rs, int32_t* tsr, void* x_packed, const Ptrs& P) {
  DispatchArgs a{};
  a.ids = ids; a.T = T; a.K = c->top_k; a.E = c->n_experts;
  a.counts = counts; a.offsets = offsets; a.route_token = rt; a.route_slot = rs; a.token_slot_row = tsr;
  a.active = P.at<int32_t>(P.L.active);
  a.hdr = P.hdr();
  a.tile_counts = P.at<int32_t>(P.L.tile_counts);
  a.tile_prefix = P.at<int32_t>(P.L.tile_prefix);
  a.tile_rows = 0;
  a.x_e = x_e; a.x_packed = x_e ? x_packed : nullptr;
  a.de = de_of(c); a.elem_bytes = act_bytes(c);
  return a;
}

moe_status_t run_dispatch(const moe_config_t* c, int T, const int32_t* ids, const void* x_e, int32_t* counts,
                          int32_t* offsets, int32_t* rt, int32_t* rs, int32_t* tsr, void* x_packed,
                          const Ptrs& P, cudaStream_t s) {
  CU(launch_dispatch(dispatch_args(c, T, ids, x_e, counts, offsets, rt, rs, tsr, x_packed, P), s));
  return MOE_OK;
}

// NVFP4 expert products multiply in FP16: the layer hands them FP16 copies of
// their BF16 input rows (exact inside FP16's range) and has the up projection
// store h as FP16 copies of its BF16 values, so no CTA converts activations
// and the tensor-core kernel's two operands share a type.  Decode needs both
// products on the streaming GEMV kernel; the tensor-core kernels always qualify.
bool up_down_f16(const moe_config_t* c, int T, const moe_weights_t* w) {
  if (c->expert_dtype != MOE_DT_NVFP4 || c->act_dtype != MOE_DT_BF16 || act_terms_for(T) > 0) return false;
  if (use_tc(c, T)) return true;
  const int de = de_of(c), I = c->d_expert;
  GemvArgs up{}, dn{};
  int32_t dummy = 0;
  up.offsets = dn.offsets = &dummy;
  up.W = w->w_up; up.W_sf = w->w_up_sf; up.N = I; up.K = de;
  dn.W = w->w_down; dn.W_sf = w->w_down_sf; dn.N = de; dn.K = I;
  return gemv_nvfp4_streams(up) && gemv_nvfp4_streams(dn);
}

// f16: x_e holds FP16 activations and h receives FP16 (the layer's NVFP4
// decode path, where up_down_f16() holds)
moe_status_t run_up_fp4(const moe_config_t* c, int T, const void* x_e, const void* x_packed, const int32_t* rt,
                        const int32_t* offsets, const moe_weights_t* w, void* h, const Ptrs& P, cudaStream_t s);
moe_status_t run_down_fp4(const moe_config_t* c, int T, const void* h, const int32_t* offsets, const int32_t* rt,
                          const int32_t* rs, const float* topw, const moe_weights_t* w, float* u, const Ptrs& P,
                          cudaStream_t s);

moe_status_t run_up(const moe_config_t* c, int T, const void* x_e, const void* x_packed, const int32_t* rt,
                    const int32_t* offsets, const moe_weights_t* w, void* h, const Ptrs& P, cudaStream_t s,
                    bool f16 = false) {
  if (fp4_path(c, T)) return run_up_fp4(c, T, x_e, x_packed, rt, offsets, w, h, P, s);
  const int de = de_of(c), I = c->d_expert;
  const bool fp4 = c->expert_dtype == MOE_DT_NVFP4;
  GemvArgs a{};
  a.W = w->w_up; a.w_seg_stride = fp4 ? (int64_t)I * de / 2 : (int64_t)I * de; a.N = I; a.K = de;
  if (fp4) { a.W_sf = w->w_up_sf; a.W_gs = w->w_up_gs; a.sf_seg_stride = (int64_t)I * de / 16; }
  a.X = x_packed ? x_packed : x_e; a.x_ld = de; a.gather = x_packed ? nullptr : rt;
  a.offsets = offsets; a.active = P.at<int32_t>(P.L.active); a.hdr = P.hdr();
  a.out = h; a.out_ld = I; a.err = &P.hdr()->err;
  a.x_f16 = a.out_f16 = f16;
  const int segs = (int)std::min<int64_t>(c->n_experts, (int64_t)T * c->top_k);
  if (use_tc(c, T)) {
    const int64_t R = (int64_t)T * c->top_k;
    if (!x_packed) {
      // the tensor-core kernel reads contiguous rows: gather them into the
      // workspace's packed-row region first
      void* xp = P.at<void>(P.L.x_packed);
      CU(launch_pack_rows(x_e, rt, offsets, c->n_experts, (int)R, de, act_bytes(c), f16, xp, s, &P.hdr()->err));
      a.X = xp;
      a.gather = nullptr;
    }
    // (NVFP4 weights are converted to BF16, or with f16 to FP16, inside the tensor-core kernel)
    CU(launch_gemm_tc(a, EPI_RELU2, false, (int64_t)c->n_experts * I, R, c->n_experts,
                      tc_tile_rows(R / segs, segs, I), s));
    return MOE_OK;
  }
  CU(launch_gemv(a, wfmt_of(c), c->act_dtype, EPI_RELU2, c->act_dtype == MOE_DT_F32, T, segs, s));
  return MOE_OK;
}

// the decode down projection runs ReLU^2-sparse up to this many tokens: above
// it too few 16-neuron groups are dead in every row of an expert (8 % at 64
// tokens of a 92.5 %-sparse Nano layer, where the sparse product measured 10 %
// slower than the dense GEMV; 16 % dead and 2 % faster at 16 tokens)
constexpr int kSparseDownMaxT = 16;

// the decode down projection can run ReLU^2-sparse: group-major weights given,
// BF16 activations, BF16 experts or NVFP4 experts with FP16 h, shapes that fit
bool sparse_down_ok(const moe_config_t* c, int T, const moe_weights_t* w, bool f16) {
  if (!w->w_down_g || c->act_dtype != MOE_DT_BF16 || T > kSparseDownMaxT) return false;
  const bool fp4 = c->expert_dtype == MOE_DT_NVFP4;
  if (fp4 && (!f16 || !w->w_down_g_sf)) return false;
  if (!fp4 && c->expert_dtype != MOE_DT_BF16) return false;
  return sparse_down_fits(de_of(c), c->d_expert, fp4);
}

moe_status_t run_down(const moe_config_t* c, int T, const void* h, const int32_t* offsets, const int32_t* rt,
                      const int32_t* rs, const float* topw, const moe_weights_t* w, float* u, const Ptrs& P,
                      cudaStream_t s, bool f16 = false) {
  if (fp4_path(c, T)) return run_down_fp4(c, T, h, offsets, rt, rs, topw, w, u, P, s);
  const int de = de_of(c), I = c->d_expert;
  const bool fp4 = c->expert_dtype == MOE_DT_NVFP4;
  GemvArgs a{};
  a.W = w->w_down; a.w_seg_stride = fp4 ? (int64_t)de * I / 2 : (int64_t)de * I; a.N = de; a.K = I;
  if (fp4) { a.W_sf = w->w_down_sf; a.W_gs = w->w_down_gs; a.sf_seg_stride = (int64_t)de * I / 16; }
  a.X = h; a.x_ld = I;
  a.offsets = offsets; a.active = P.at<int32_t>(P.L.active); a.hdr = P.hdr();
  a.out = u; a.out_ld = de;
  a.topw = topw; a.route_token = rt; a.route_slot = rs; a.top_k = c->top_k; a.err = &P.hdr()->err;
  a.x_f16 = f16;
  const int segs = (int)std::min<int64_t>(c->n_experts, (int64_t)T * c->top_k);
  if (use_tc(c, T)) {
    const int64_t R = (int64_t)T * c->top_k;
    CU(launch_gemm_tc(a, EPI_SCALE, true, (int64_t)c->n_experts * de, R, c->n_experts,
                      tc_tile_rows(R / segs, segs, de), s));
    return MOE_OK;
  }
  if (sparse_down_ok(c, T, w, f16)) {
    // ReLU^2-sparse: only the 16-neuron groups of W_down with a live neuron
    a.W = w->w_down_g;
    a.W_sf = w->w_down_g_sf;
    CU(launch_sparse_down(a, fp4, segs, s));
    return MOE_OK;
  }
  CU(launch_gemv(a, wfmt_of(c), c->act_dtype, EPI_SCALE, true, T, segs, s));
  return MOE_OK;
}

// ---- NVFP4 experts on the FP4 tensor path ----
inline bool fp4_path(const moe_config_t* c, int T) { return c->expert_dtype == MOE_DT_NVFP4 && act_terms_for(T) > 0; }

// packed rows per tile of an expert product with N output features (a decode
// tile holds an expert's rows)
inline int fp4_bn(const moe_config_t* c, int T, int N) {
  const int64_t R = (int64_t)T * c->top_k;
  const int64_t segs = std::min<int64_t>(c->n_experts, R);
  return fp4_tile_rows(ceil_div(R, std::max<int64_t>(segs, 1)), segs, N);
}

// grouped FP4 product: W (NVFP4, [E, N, K]) times the NVFP4 terms of the
// packed rows in q / q_sf / q_g
GemvArgs fp4_args(const moe_config_t* c, int T, const void* W, const uint8_t* W_sf, const float* W_gs, int N, int K,
                  const uint8_t* q, const uint8_t* q_sf, const float* q_g, const int32_t* offsets, int nt,
                  const Ptrs& P) {
  GemvArgs a{};
  a.W = W; a.W_sf = W_sf; a.W_gs = W_gs; a.N = N; a.K = K;
  a.X = q; a.X_sf = q_sf; a.x_scale = q_g; a.x_sf_ld = act_sf_ld(K);
  a.x_rows_cap = (int64_t)T * c->top_k; a.x_terms = nt;
  a.offsets = offsets; a.active = P.at<int32_t>(P.L.active); a.hdr = P.hdr(); a.err = &P.hdr()->err;
  return a;
}

// h = bf16(relu(bf16(x_e W_up^T))^2) for every packed row: the rows (x_packed,
// or x_e gathered through rt) become NVFP4 terms, then the FP4 product
moe_status_t run_up_fp4(const moe_config_t* c, int T, const void* x_e, const void* x_packed, const int32_t* rt,
                        const int32_t* offsets, const moe_weights_t* w, void* h, const Ptrs& P, cudaStream_t s) {
  const int de = de_of(c), I = c->d_expert, nt = act_terms_for(T);
  const int R = T * c->top_k;
  uint8_t* xq = P.at<uint8_t>(P.L.xq);
  uint8_t* xq_sf = P.at<uint8_t>(P.L.xq_sf);
  float* xq_g = P.at<float>(P.L.xq_g);
  const void* src = x_packed ? x_packed : x_e;
  CU(launch_quant_terms(src, de, x_packed ? nullptr : rt, offsets + c->n_experts, R, de, nt, xq, xq_sf, xq_g, R, s));
  GemvArgs a = fp4_args(c, T, w->w_up, w->w_up_sf, w->w_up_gs, I, de, xq, xq_sf, xq_g, offsets, nt, P);
  a.out = h; a.out_ld = I;
  CU(launch_gemm_fp4(a, EPI_RELU2, false, (int64_t)c->n_experts * I, c->n_experts, fp4_bn(c, T, I), s));
  return MOE_OK;
}

// u = w * (h W_down^T) for every packed row (FP32), h quantised to NVFP4 terms first
moe_status_t run_down_fp4(const moe_config_t* c, int T, const void* h, const int32_t* offsets, const int32_t* rt,
                          const int32_t* rs, const float* topw, const moe_weights_t* w, float* u, const Ptrs& P,
                          cudaStream_t s) {
  const int de = de_of(c), I = c->d_expert, nt = act_terms_for(T);
  const int R = T * c->top_k;
  uint8_t* hq = P.at<uint8_t>(P.L.hq);
  uint8_t* hq_sf = P.at<uint8_t>(P.L.hq_sf);
  float* hq_g = P.at<float>(P.L.hq_g);
  CU(launch_quant_terms(h, I, nullptr, offsets + c->n_experts, R, I, nt, hq, hq_sf, hq_g, R, s));
  GemvArgs a = fp4_args(c, T, w->w_down, w->w_down_sf, w->w_down_gs, de, I, hq, hq_sf, hq_g, offsets, nt, P);
  a.out = u; a.out_ld = de;
  a.topw = topw; a.route_token = rt; a.route_slot = rs; a.top_k = c->top_k;
  CU(launch_gemm_fp4(a, EPI_SCALE, true, (int64_t)c->n_experts * de, c->n_experts, fp4_bn(c, T, de), s));
  return MOE_OK;
}

moe_status_t run_latent_down(const moe_config_t* c, int T, const void* x, const moe_weights_t* w, void* x_l,
                             cudaStream_t s) {
  GemvArgs a = dense_args(w->w_lat_down, c->d_latent, c->d_model, x, T, x_l, c->d_latent);
  CU(run_dense(c, a, EPI_STORE, false, T, s));
  return MOE_OK;
}

// shared expert + output; y_rl = act-typed routed latent rows (latent shapes, may be null)
moe_status_t run_shared(const moe_config_t* c, int T, const void* x, const moe_weights_t* w, const float* y_r,
                        const void* y_rl, void* y, const Ptrs& P, cudaStream_t s) {
  const int d = c->d_model, S = c->d_shared;
  const bool latent = c->d_latent > 0;
  const bool f32 = c->act_dtype == MOE_DT_F32;
  if (S > 0) {
    void* hs = P.at<void>(P.L.hs);
    GemvArgs up = dense_args(w->w_sh_up, S, d, x, T, hs, S);
    CU(run_dense(c, up, EPI_RELU2, f32, T, s));
    GemvArgs dn = dense_args(w->w_sh_down, d, S, hs, T, nullptr, d);
    if (!latent) {
      dn.out = y; dn.add_src = y_r; dn.add_ld = d;
      CU(run_dense(c, dn, EPI_ADD, f32, T, s));
      return MOE_OK;
    }
    dn.out = P.at<void>(P.L.ys);
    CU(run_dense(c, dn, EPI_STORE, true, T, s));
  } else if (!latent) {
    // no shared expert: y = act(y_r); a combine over one row per token is a cast
    CU(launch_cast(y_r, (int64_t)T * d, y, c->act_dtype, s));
    return MOE_OK;
  }
  // latent up: y = act(act(y_r) W_lu^T + y_s)
  const void* yl = y_rl;
  if (!yl) {
    void* tmp = P.at<void>(P.L.y_rl);
    CU(launch_cast(y_r, (int64_t)T * c->d_latent, tmp, c->act_dtype, s));
    yl = tmp;
  }
  GemvArgs lu = dense_args(w->w_lat_up, d, c->d_latent, yl, T, y, d);
  lu.add_src = S > 0 ? P.at<float>(P.L.ys) : nullptr;
  lu.add_ld = d;
  CU(run_dense(c, lu, EPI_ADD, f32, T, s));
  return MOE_OK;
}

// One auxiliary stream and a fork/join event pair per device, created on first
// use: moe_layer_forward runs the shared expert there, concurrently with the
// router -> dispatch -> experts chain on the caller's stream.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, latent = nullptr;
};
std::mutex g_aux_mutex;
AuxStream g_aux[kMaxDevices];

bool aux_stream(AuxStream** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  AuxStream& a = g_aux[dev];
  if (!a.s) {
    if (cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&a.latent, cudaEventDisableTiming) != cudaSuccess) return false;
  }
  *out = &a;
  return true;
}

// shared expert y_s[T, d] (FP32) = W_sd act(relu(act(W_su x))^2)
moe_status_t run_shared_to_f32(const moe_config_t* c, int T, const void* x, const moe_weights_t* w, float* ys,
                               const Ptrs& P, cudaStream_t s) {
  const int d = c->d_model, S = c->d_shared;
  const bool f32 = c->act_dtype == MOE_DT_F32;
  void* hs = P.at<void>(P.L.hs);
  GemvArgs up = dense_args(w->w_sh_up, S, d, x, T, hs, S);
  CU(run_dense(c, up, EPI_RELU2, f32, T, s));
  GemvArgs dn = dense_args(w->w_sh_down, d, S, hs, T, ys, d);
  CU(run_dense(c, dn, EPI_STORE, true, T, s));
  return MOE_OK;
}

moe_status_t check_weights(const moe_config_t* c, const moe_weights_t* w, bool experts, bool router, bool dense) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (router) { REQ(w->w_router); OPT(w->router_bias); }
  if (experts) {
    REQ(w->w_up); REQ(w->w_down);
    if (c->expert_dtype == MOE_DT_NVFP4) {
      if (!w->w_up_sf || !w->w_down_sf) return MOE_ERR_INVALID_ARG;
      REQ(w->w_up_gs); REQ(w->w_down_gs);
      if (((uintptr_t)w->w_up_sf & 1u) || ((uintptr_t)w->w_down_sf & 1u)) return MOE_ERR_INVALID_ARG;
    }
  }
  if (experts) { OPT(w->w_down_g); OPT(w->w_down_g_sf); }
  if (dense) {
    if (c->d_latent > 0) { REQ(w->w_lat_down); REQ(w->w_lat_up); }
    if (c->d_shared > 0) { REQ(w->w_sh_up); REQ(w->w_sh_down); }
  }
  return MOE_OK;
}

// The layer on the caller's stream after the workspace header is cleared:
// y = act(layer(x) + resid) (resid: the block's residual rows in the
// activation type, or nullptr; y may be resid itself).
moe_status_t run_layer(const moe_config_t* cfg, int32_t T, const void* x, const void* resid, const moe_weights_t* w,
                       void* y, int32_t* topk_ids_out, float* topk_w_out, float* logits_out, float* scores_out,
                       const Ptrs& P, cudaStream_t s) {
  moe_status_t st = MOE_OK;
  // fork: the latent down projection and the shared expert run on the
  // auxiliary stream, the router and the selection on the caller's stream
  const bool shared = cfg->d_shared > 0;
  const bool latent = cfg->d_latent > 0;
  float* ys = P.at<float>(P.L.ys);
  const void* x_e = latent ? P.at<void>(P.L.x_l) : x;
  // NVFP4: FP16 expert rows; decode makes an FP16 copy of x_e in the (then
  // unused) packed-row buffer, prefill packs the rows as FP16
  const bool f16 = up_down_f16(cfg, T, w);
  const bool conv = f16 && !use_tc(cfg, T);
  void* x16 = conv ? P.at<void>(P.L.x_packed) : nullptr;
  const bool pre = latent || conv;         // work before the expert up projection
  std::unique_lock<std::mutex> aux_lock(g_aux_mutex);
  AuxStream* aux = nullptr;
  if (shared || pre) {
    if (!aux_stream(&aux)) return MOE_ERR_CUDA;
    CU(cudaEventRecord(aux->fork, s));
    CU(cudaStreamWaitEvent(aux->s, aux->fork, 0));
    if (latent && (st = run_latent_down(cfg, T, x, w, const_cast<void*>(x_e), aux->s)) != MOE_OK) return st;
    if (conv) CU(launch_bf16_to_f16(x_e, (int64_t)T * de_of(cfg), x16, aux->s, &P.hdr()->err));
    if (pre) CU(cudaEventRecord(aux->latent, aux->s));
    if (shared && (st = run_shared_to_f32(cfg, T, x, w, ys, P, aux->s)) != MOE_OK) return st;
    CU(cudaEventRecord(aux->join, aux->s));
  }
  // the lock stays held until this call's waits on the fork/latent/join events
  // are enqueued on the caller's stream (at return): another thread cannot
  // re-record the events in between
  float* logits = logits_out ? logits_out : P.at<float>(P.L.logits);
  float* scores = scores_out ? scores_out : P.at<float>(P.L.scores);
  int32_t* ids = topk_ids_out ? topk_ids_out : P.at<int32_t>(P.L.ids);
  float* topw = topk_w_out ? topk_w_out : P.at<float>(P.L.topw);
  SelectArgs sa;
  if ((st = run_logits(cfg, T, x, w->w_router, w->router_bias, logits, scores, ids, topw, P, s, sa)) != MOE_OK)
    return st;
  int32_t* offsets = P.at<int32_t>(P.L.offsets);
  int32_t* rt = P.at<int32_t>(P.L.route_token);
  int32_t* rs = P.at<int32_t>(P.L.route_slot);
  int32_t* tsr = P.at<int32_t>(P.L.tsr);
  void* x_packed = use_tc(cfg, T) && !fp4_path(cfg, T) ? P.at<void>(P.L.x_packed) : nullptr;
  DispatchArgs da = dispatch_args(cfg, T, ids, x_e, P.at<int32_t>(P.L.counts), offsets, rt, rs, tsr, x_packed, P);
  da.pack_f16 = f16 && x_packed;
  if (select_dispatch_fits(T, cfg->top_k, da)) {
    CU(launch_select_dispatch(sa, da, s));       // a few tokens: one kernel
  } else {
    CU(launch_select(sa, s));
    if (latent && x_packed) CU(cudaStreamWaitEvent(s, aux->latent, 0));   // the pack reads the latent rows
    CU(launch_dispatch(da, s));
  }
  if (pre && !x_packed) CU(cudaStreamWaitEvent(s, aux->latent, 0));    // the up GEMV reads them
  void* h = P.at<void>(P.L.h);
  if ((st = run_up(cfg, T, conv ? x16 : x_e, x_packed, rt, offsets, w, h, P, s, f16)) != MOE_OK) return st;
  float* u = P.at<float>(P.L.u);
  if ((st = run_down(cfg, T, h, offsets, rt, rs, topw, w, u, P, s, f16)) != MOE_OK) return st;
  if (cfg->d_latent == 0) {
    // join, then y = act(sum of routed rows + y_s): the same two FP32 terms, one rounding
    if (aux) CU(cudaStreamWaitEvent(s, aux->join, 0));
    CU(launch_combine(u, tsr, T, cfg->top_k, de_of(cfg), nullptr, y, cfg->act_dtype, s, shared ? ys : nullptr,
                      resid));
    return MOE_OK;
  }
  // latent: combined latent rows rounded once, then latent up + y_s
  void* y_rl = P.at<void>(P.L.y_rl);
  CU(launch_combine(u, tsr, T, cfg->top_k, de_of(cfg), nullptr, y_rl, cfg->act_dtype, s));
  if (aux) CU(cudaStreamWaitEvent(s, aux->join, 0));
  GemvArgs lu = dense_args(w->w_lat_up, cfg->d_model, cfg->d_latent, y_rl, T, y, cfg->d_model);
  lu.add_src = shared ? ys : nullptr;
  lu.add_ld = cfg->d_model;
  lu.res = resid;
  lu.res_ld = cfg->d_model;
  CU(run_dense(cfg, lu, EPI_ADD, cfg->act_dtype == MOE_DT_F32, T, s));
  return MOE_OK;
}

// ---- backward ----------------------------------------------------------------
// backward scratch [T tokens]: bf16 and f32 intermediates of moe_layer_backward
struct BwLayout {
  size_t tprefix, dyr, dU, q, dz, da, dxr, dxe, dxl, das, dxs, dxa, dxn, xr, total;
};

BwLayout make_bw_layout(const moe_config_t* c, int32_t T) {
  BwLayout B{};
  const size_t t = (size_t)T, R = t * c->top_k, de = de_of(c), d = c->d_model, I = c->d_expert;
  const size_t S = c->d_shared, L = c->d_latent;
  size_t off = 0;
  B.tprefix = take(off, ((size_t)c->n_experts + 1) * 4);
  B.dyr = take(off, L ? t * L * 2 : 0);
  B.dU = take(off, R * de * 2);
  B.q = take(off, R * 4);
  B.dz = take(off, R * 4);
  B.da = take(off, R * I * 2);
  B.dxr = take(off, R * de * 4);
  B.dxe = take(off, t * de * 4);
  B.dxl = take(off, L ? t * L * 2 : 0);
  B.das = take(off, t * S * 2);
  B.dxs = take(off, S ? t * d * 4 : 0);
  B.dxa = take(off, L ? t * d * 4 : 0);
  B.dxn = take(off, t * d * 4);
  B.xr = take(off, t * d * 4);
  B.total = (off + 255) & ~(size_t)255;
  return B;
}

moe_status_t check_backward(const moe_config_t* c, int32_t T, const void* ws, size_t ws_bytes, const void* bws,
                            size_t bws_bytes) {
  moe_status_t st = check_common(c, T, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (c->act_dtype != MOE_DT_BF16 || c->expert_dtype != MOE_DT_BF16) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!bws || !aligned16(bws)) return MOE_ERR_INVALID_ARG;
  if (bws_bytes < make_bw_layout(c, T).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// one backward GEMM's arguments
GemmArgs gemm_args(int mode, int epi, const void* A, int64_t lda, bool a_t, const void* B, int64_t ldb, void* C,
                   int64_t ldc, int M, int N, int K) {
  GemmArgs g{};
  g.mode = mode; g.epi = epi;
  g.A = reinterpret_cast<const bf16*>(A); g.lda = lda; g.a_t = a_t;
  g.B = reinterpret_cast<const bf16*>(B); g.ldb = ldb;
  g.C = C; g.ldc = ldc;
  g.M = M; g.N = N; g.K = K;
  return g;
}

// Gradients of L = <dy, y> for the layer whose forward on x left its route
// tables, h, u, the latent rows, y_rl and the shared h in P (no other layer
// call on that workspace since).  dx (FP32) is written; weight gradients are
// added to g's non-NULL buffers.
moe_status_t run_backward(const moe_config_t* c, int T, const void* x, const moe_weights_t* w, const void* dy,
                          const int32_t* ids, const float* topw, const float* scores, float* dx,
                          const moe_grads_t* gr, const Ptrs& P, char* bws, cudaStream_t s) {
  const BwLayout B = make_bw_layout(c, T);
  auto at = [&](size_t o) { return bws + o; };
  const int d = c->d_model, de = de_of(c), I = c->d_expert, S = c->d_shared, L = c->d_latent;
  const int E = c->n_experts, K = c->top_k, R = T * K;
  const bool latent = L > 0, shared = S > 0;
  const int segs = (int)std::min<int64_t>(E, R);
  const int32_t* offs = P.at<int32_t>(P.L.offsets);
  const int32_t* active = P.at<int32_t>(P.L.active);
  const int32_t* rt = P.at<int32_t>(P.L.route_token);
  const int32_t* rs = P.at<int32_t>(P.L.route_slot);
  const int32_t* tsr = P.at<int32_t>(P.L.tsr);
  const WsHeader* hdr = P.hdr();
  const void* x_e = latent ? P.at<void>(P.L.x_l) : x;
  int32_t* tpre = reinterpret_cast<int32_t*>(at(B.tprefix));
  auto grouped = [&](GemmArgs& g) {
    g.offsets = offs; g.active = active; g.hdr = hdr; g.tprefix = tpre;
  };
  CU(launch_tile_scan(offs, active, hdr, tpre, s));
  // upstream gradient of the routed sum: dy, or dy W_lu (latent)
  const void* dyr = dy;
  int64_t dyr_ld = d;
  if (latent) {
    GemmArgs g = gemm_args(GM_ROWS, GE_STORE_BF16, dy, d, false, w->w_lat_up, L, at(B.dyr), L, 0, L, d);
    g.dense_rows = T;
    CU(launch_gemm_bwd(g, 1, T, s));
    if (gr->d_lat_up) {
      // dW_lu += dy^T y_rl  (y_rl: the forward's rounded latent combine)
      GemmArgs gw = gemm_args(GM_KSEG, GE_ACC_F32, dy, d, true, P.at<void>(P.L.y_rl), L, gr->d_lat_up, L, d, L, 0);
      gw.dense_rows = T;
      CU(launch_gemm_bwd(gw, 1, 0, s));
    }
    dyr = at(B.dyr);
    dyr_ld = L;
  }
  // combine backward: dU = w dy_r (packed rows), q = <dy_r, U>
  CU(launch_combine_bwd(dyr, dyr_ld, P.at<float>(P.L.u), rt, rs, topw, R, K, de, at(B.dU),
                        reinterpret_cast<float*>(at(B.q)), s));
  // gate backward and the router weight gradient
  float* dz = reinterpret_cast<float*>(at(B.dz));
  CU(launch_gate_bwd(scores, ids, reinterpret_cast<float*>(at(B.q)), T, E, K, c->norm_topk_prob,
                     c->routed_scaling_factor, dz, s));
  if (gr->d_router)
    CU(launch_router_wgrad(x, false, d, dz, rt, rs, K, offs, active, hdr, segs, gr->d_router, s));
  // experts: da = (dU W_down,e) * 2 relu(a);  dW_down,e += dU^T h;  dW_up,e += da^T x_e;  dx_e rows = da W_up,e
  {
    GemmArgs g = gemm_args(GM_ROWS, GE_RELU2_GRAD, at(B.dU), de, false, w->w_down, I, at(B.da), I, 0, I, de);
    g.b_seg = (int64_t)de * I;
    g.aux = P.at<bf16>(P.L.h);
    g.aux_ld = I;
    grouped(g);
    CU(launch_gemm_bwd(g, segs, R, s));
  }
  if (gr->d_down) {
    GemmArgs g = gemm_args(GM_KSEG, GE_ACC_F32, at(B.dU), de, true, P.at<void>(P.L.h), I, gr->d_down, I, de, I, 0);
    g.c_seg = (int64_t)de * I;
    grouped(g);
    CU(launch_gemm_bwd(g, segs, 0, s));
  }
  if (gr->d_up) {
    GemmArgs g = gemm_args(GM_KSEG, GE_ACC_F32, at(B.da), I, true, x_e, de, gr->d_up, de, I, de, 0);
    g.c_seg = (int64_t)I * de;
    g.b_gather = rt;
    grouped(g);
    CU(launch_gemm_bwd(g, segs, 0, s));
  }
  {
    GemmArgs g = gemm_args(GM_ROWS, GE_STORE_F32, at(B.da), I, false, w->w_up, de, at(B.dxr), de, 0, de, I);
    g.b_seg = (int64_t)I * de;
    grouped(g);
    CU(launch_gemm_bwd(g, segs, R, s));
  }
  // scatter-add of the routed rows' input gradients to their tokens, in
  // ascending packed row (= expert) order (the combine's own order)
  float* dxe = reinterpret_cast<float*>(at(B.dxe));
  CU(launch_combine(reinterpret_cast<float*>(at(B.dxr)), tsr, T, K, de, dxe, latent ? at(B.dxl) : nullptr,
                    MOE_DT_BF16, s));
  const float* dx_expert = dxe;
  if (latent) {
    // dW_ld += dx_l^T x;  dx_latent = dx_l W_ld   (dx_l rounded to BF16 for the products)
    if (gr->d_lat_down) {
      GemmArgs gw = gemm_args(GM_KSEG, GE_ACC_F32, at(B.dxl), L, true, x, d, gr->d_lat_down, d, L, d, 0);
      gw.dense_rows = T;
      CU(launch_gemm_bwd(gw, 1, 0, s));
    }
    GemmArgs g = gemm_args(GM_ROWS, GE_STORE_F32, at(B.dxl), L, false, w->w_lat_down, d, at(B.dxa), d, 0, d, L);
    g.dense_rows = T;
    CU(launch_gemm_bwd(g, 1, T, s));
    dx_expert = reinterpret_cast<float*>(at(B.dxa));
  }
  const float* dx_shared = nullptr;
  if (shared) {
    // da_s = (dy W_sd) * 2 relu(a_s);  dW_sd += dy^T h_s;  dW_su += da_s^T x;  dx_s = da_s W_su
    GemmArgs g = gemm_args(GM_ROWS, GE_RELU2_GRAD, dy, d, false, w->w_sh_down, S, at(B.das), S, 0, S, d);
    g.dense_rows = T;
    g.aux = P.at<bf16>(P.L.hs);
    g.aux_ld = S;
    CU(launch_gemm_bwd(g, 1, T, s));
    if (gr->d_sh_down) {
      GemmArgs gw = gemm_args(GM_KSEG, GE_ACC_F32, dy, d, true, P.at<void>(P.L.hs), S, gr->d_sh_down, S, d, S, 0);
      gw.dense_rows = T;
      CU(launch_gemm_bwd(gw, 1, 0, s));
    }
    if (gr->d_sh_up) {
      GemmArgs gw = gemm_args(GM_KSEG, GE_ACC_F32, at(B.das), S, true, x, d, gr->d_sh_up, d, S, d, 0);
      gw.dense_rows = T;
      CU(launch_gemm_bwd(gw, 1, 0, s));
    }
    GemmArgs g2 = gemm_args(GM_ROWS, GE_STORE_F32, at(B.das), S, false, w->w_sh_up, d, at(B.dxs), d, 0, d, S);
    g2.dense_rows = T;
    CU(launch_gemm_bwd(g2, 1, T, s));
    dx_shared = reinterpret_cast<float*>(at(B.dxs));
  }
  // dx = router path + expert path + shared path
  CU(launch_input_grad(dz, ids, T, K, w->w_router, d, dx_expert, dx_shared, dx, s));
  return MOE_OK;
}

}  // namespace

// ============================================================================
extern "C" {

int32_t moe_version(void) { return 100; }

int64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device-side error flag set";
    default: return "unknown status";
  }
}

moe_status_t moe_check_config(const moe_config_t* cfg) { return check_config(cfg); }

int32_t moe_nvfp4_act_terms_for(int32_t T) { return act_terms_for(T); }

int32_t moe_set_nvfp4_act_terms(int32_t n) {
  if (n < -1 || n > kActTermsMax) return -2;
  return g_act_terms.exchange(n);
}

moe_status_t moe_workspace_region(const moe_config_t* cfg, int32_t T, int32_t region, size_t* offset,
                                  size_t* bytes) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (T < 0 || !offset || !bytes) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(cfg, T);
  const size_t t = (size_t)T, E = cfg->n_experts, R = t * cfg->top_k;
  const size_t ab = act_bytes(cfg);
  const bool fp4 = cfg->expert_dtype == MOE_DT_NVFP4;
  const size_t nt = fp4 ? kActTermsMax : 0, de = de_of(cfg), I = cfg->d_expert;
  size_t o = 0, n = 0;
  switch (region) {
    case MOE_WS_COUNTS: o = L.counts; n = E * 4; break;
    case MOE_WS_OFFSETS: o = L.offsets; n = (E + 1) * 4; break;
    case MOE_WS_ROUTE_TOKEN: o = L.route_token; n = R * 4; break;
    case MOE_WS_ROUTE_SLOT: o = L.route_slot; n = R * 4; break;
    case MOE_WS_TOKEN_SLOT_ROW: o = L.tsr; n = R * 4; break;
    case MOE_WS_TOPK_IDS: o = L.ids; n = R * 4; break;
    case MOE_WS_TOPK_W: o = L.topw; n = R * 4; break;
    case MOE_WS_LOGITS: o = L.logits; n = t * E * 4; break;
    case MOE_WS_SCORES: o = L.scores; n = t * E * 4; break;
    case MOE_WS_X_LATENT: o = L.x_l; n = t * (size_t)cfg->d_latent * ab; break;
    case MOE_WS_X_PACKED: o = L.x_packed; n = R * (size_t)de_of(cfg) * ab; break;
    case MOE_WS_H: o = L.h; n = R * (size_t)cfg->d_expert * ab; break;
    case MOE_WS_X_TERMS: o = L.xq; n = nt * R * de / 2; break;
    case MOE_WS_X_TERM_SCALES: o = L.xq_sf; n = nt * R * (size_t)act_sf_ld((int)de); break;
    case MOE_WS_X_ROW_SCALES: o = L.xq_g; n = fp4 ? R * 4 : 0; break;
    case MOE_WS_H_TERMS: o = L.hq; n = nt * R * I / 2; break;
    case MOE_WS_H_TERM_SCALES: o = L.hq_sf; n = nt * R * (size_t)act_sf_ld((int)I); break;
    case MOE_WS_H_ROW_SCALES: o = L.hq_g; n = fp4 ? R * 4 : 0; break;
    case MOE_WS_X_NORM: o = L.xn; n = t * (size_t)cfg->d_model * ab; break;
    default: return MOE_ERR_INVALID_ARG;
  }
  *offset = o;
  *bytes = n;
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_config_t* cfg, int32_t T) {
  if (check_config(cfg) != MOE_OK || T < 0) return 0;
  return make_layout(cfg, T).total;
}

moe_status_t moe_router(const moe_config_t* cfg, int32_t T, const void* x, const float* w_router,
                        const float* router_bias, float* logits, float* scores, int32_t* topk_ids, float* topk_w,
                        void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  REQ(x); REQ(w_router); OPT(router_bias); OPT(logits); OPT(scores); REQ(topk_ids); REQ(topk_w);
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  return run_router(cfg, T, x, w_router, router_bias, logits ? logits : P.at<float>(P.L.logits),
                    scores ? scores : P.at<float>(P.L.scores), topk_ids, topk_w, P, (cudaStream_t)stream);
}

moe_status_t moe_dispatch(const moe_config_t* cfg, int32_t T, const int32_t* topk_ids, const void* x_e,
                          int32_t* counts, int32_t* offsets, int32_t* route_token, int32_t* route_slot,
                          int32_t* token_slot_row, void* x_packed, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  REQ(topk_ids); OPT(x_e); REQ(counts); REQ(offsets); REQ(route_token); REQ(route_slot); REQ(token_slot_row);
  OPT(x_packed);
  if (x_packed && !x_e) return MOE_ERR_INVALID_ARG;
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  return run_dispatch(cfg, T, topk_ids, x_e, counts, offsets, route_token, route_slot, token_slot_row, x_packed,
                      P, (cudaStream_t)stream);
}

moe_status_t moe_experts_up(const moe_config_t* cfg, int32_t T, const void* x_e, const void* x_packed,
                            const int32_t* route_token, const int32_t* offsets, const moe_weights_t* w, void* h,
                            void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, false, false)) != MOE_OK) return st;
  OPT(x_e); OPT(x_packed); REQ(route_token); REQ(offsets); REQ(h);
  if (!x_e && !x_packed) return MOE_ERR_INVALID_ARG;
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  return run_up(cfg, T, x_e, x_packed, route_token, offsets, w, h, P, (cudaStream_t)stream);
}

moe_status_t moe_experts_down_combine(const moe_config_t* cfg, int32_t T, const void* h, const int32_t* offsets,
                                      const int32_t* route_token, const int32_t* route_slot,
                                      const int32_t* token_slot_row, const float* topk_w, const moe_weights_t* w,
                                      float* y_routed, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, false, false)) != MOE_OK) return st;
  REQ(h); REQ(offsets); REQ(route_token); REQ(route_slot); REQ(token_slot_row); REQ(topk_w); REQ(y_routed);
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  cudaStream_t s = (cudaStream_t)stream;
  float* u = P.at<float>(P.L.u);
  if ((st = run_down(cfg, T, h, offsets, route_token, route_slot, topk_w, w, u, P, s)) != MOE_OK) return st;
  CU(launch_combine(u, token_slot_row, T, cfg->top_k, de_of(cfg), y_routed, nullptr, cfg->act_dtype, s));
  return MOE_OK;
}

moe_status_t moe_experts_down(const moe_config_t* cfg, int32_t T, const void* h, const int32_t* offsets,
                              const int32_t* route_token, const int32_t* route_slot, const float* topk_w,
                              const moe_weights_t* w, float* u, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, false, false)) != MOE_OK) return st;
  REQ(h); REQ(offsets); REQ(route_token); REQ(route_slot); REQ(topk_w); REQ(u);
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  return run_down(cfg, T, h, offsets, route_token, route_slot, topk_w, w, u, P, (cudaStream_t)stream);
}

moe_status_t moe_latent_down(const moe_config_t* cfg, int32_t T, const void* x, const moe_weights_t* w, void* x_l,
                             void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if (cfg->d_latent <= 0) return MOE_ERR_INVALID_ARG;
  if (!w) return MOE_ERR_INVALID_ARG;
  REQ(x); REQ(w->w_lat_down); REQ(x_l);
  return run_latent_down(cfg, T, x, w, x_l, (cudaStream_t)stream);
}

moe_status_t moe_shared(const moe_config_t* cfg, int32_t T, const void* x, const moe_weights_t* w,
                        const float* y_routed, void* y, void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, false, false, true)) != MOE_OK) return st;
  REQ(x); OPT(y_routed); REQ(y);
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  cudaStream_t s = (cudaStream_t)stream;
  const float* yr = y_routed;
  if (!yr) {
    // no routed output: treat as zero
    float* z = P.at<float>(P.L.y_r);
    CU(cudaMemsetAsync(z, 0, (size_t)T * de_of(cfg) * 4, s));
    yr = z;
  }
  return run_shared(cfg, T, x, w, yr, nullptr, y, P, s);
}

moe_status_t moe_layer_forward(const moe_config_t* cfg, int32_t T, const void* x, const moe_weights_t* w, void* y,
                               int32_t* topk_ids_out, float* topk_w_out, float* logits_out, float* scores_out,
                               void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, true, true)) != MOE_OK) return st;
  REQ(x); REQ(y); OPT(topk_ids_out); OPT(topk_w_out); OPT(logits_out); OPT(scores_out);
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  cudaStream_t s = (cudaStream_t)stream;
  CU(cudaMemsetAsync(P.hdr(), 0, sizeof(WsHeader), s));
  return run_layer(cfg, T, x, nullptr, w, y, topk_ids_out, topk_w_out, logits_out, scores_out, P, s);
}

moe_status_t moe_sparse_down_bytes(const moe_config_t* cfg, size_t* values, size_t* scales) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!values || !scales) return MOE_ERR_INVALID_ARG;
  const bool fp4 = cfg->expert_dtype == MOE_DT_NVFP4;
  if (cfg->act_dtype != MOE_DT_BF16 || !sparse_down_fits(de_of(cfg), cfg->d_expert, fp4))
    return MOE_ERR_UNSUPPORTED;
  const size_t n = (size_t)cfg->n_experts * de_of(cfg) * cfg->d_expert;
  *values = fp4 ? n / 2 : n * 2;
  *scales = fp4 ? n / 16 : 0;
  return MOE_OK;
}

moe_status_t moe_sparse_down_layout(const moe_config_t* cfg, const moe_weights_t* w, void* w_down_g,
                                    uint8_t* w_down_g_sf, void* stream) {
  size_t nv = 0, ns = 0;
  moe_status_t st = moe_sparse_down_bytes(cfg, &nv, &ns);
  if (st != MOE_OK) return st;
  if (!w) return MOE_ERR_INVALID_ARG;
  const bool fp4 = cfg->expert_dtype == MOE_DT_NVFP4;
  REQ(w->w_down); REQ(w_down_g);
  if (fp4) { REQ(w->w_down_sf); REQ(w_down_g_sf); }
  CU(launch_sparse_down_layout(w->w_down, fp4 ? w->w_down_sf : nullptr, cfg->n_experts, de_of(cfg),
                               cfg->d_expert, fp4, w_down_g, fp4 ? w_down_g_sf : nullptr,
                               (cudaStream_t)stream));
  return MOE_OK;
}

moe_status_t moe_block_forward(const moe_config_t* cfg, int32_t T, const void* x, const float* norm_w,
                               float norm_eps, const moe_weights_t* w, void* out, void* x_norm_out,
                               int32_t* topk_ids_out, float* topk_w_out, float* logits_out, float* scores_out,
                               void* ws, size_t ws_bytes, void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, true, true)) != MOE_OK) return st;
  REQ(x); REQ(norm_w); REQ(out); OPT(x_norm_out); OPT(topk_ids_out); OPT(topk_w_out); OPT(logits_out);
  OPT(scores_out);
  if (!std::isfinite(norm_eps) || norm_eps < 0.f) return MOE_ERR_INVALID_ARG;
  Ptrs P{(char*)ws, make_layout(cfg, T)};
  const size_t row_bytes = (size_t)T * cfg->d_model * act_bytes(cfg);
  if (x_norm_out) {
    // the normalised rows must not overlap the residual stream
    const char *a = (const char*)x_norm_out, *b = (const char*)x, *o = (const char*)out;
    if ((a < b + row_bytes && b < a + row_bytes) || (a < o + row_bytes && o < a + row_bytes))
      return MOE_ERR_INVALID_ARG;
  }
  if (out != x) {
    const char *b = (const char*)x, *o = (const char*)out;
    if (b < o + row_bytes && o < b + row_bytes) return MOE_ERR_INVALID_ARG;   // partial overlap
  }
  cudaStream_t s = (cudaStream_t)stream;
  void* xn = x_norm_out ? x_norm_out : P.at<void>(P.L.xn);
  CU(launch_rmsnorm(x, norm_w, norm_eps, T, cfg->d_model, cfg->act_dtype, xn, P.hdr(), (int)sizeof(WsHeader), s));
  return run_layer(cfg, T, xn, x, w, out, topk_ids_out, topk_w_out, logits_out, scores_out, P, s);
}

size_t moe_backward_workspace_bytes(const moe_config_t* cfg, int32_t T) {
  if (check_config(cfg) != MOE_OK || T < 0) return 0;
  return make_bw_layout(cfg, T).total;
}

moe_status_t moe_backward_workspace_region(const moe_config_t* cfg, int32_t T, int32_t region, size_t* offset,
                                           size_t* bytes) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (T < 0 || !offset || !bytes) return MOE_ERR_INVALID_ARG;
  const BwLayout B = make_bw_layout(cfg, T);
  const size_t t = (size_t)T, R = t * cfg->top_k, de = de_of(cfg), I = cfg->d_expert;
  size_t o = 0, n = 0;
  switch (region) {
    case MOE_BWS_DU: o = B.dU; n = R * de * 2; break;
    case MOE_BWS_DA: o = B.da; n = R * I * 2; break;
    case MOE_BWS_DZ: o = B.dz; n = R * 4; break;
    case MOE_BWS_DX_LATENT: o = B.dxl; n = cfg->d_latent ? t * cfg->d_latent * 2 : 0; break;
    case MOE_BWS_DA_SHARED: o = B.das; n = t * (size_t)cfg->d_shared * 2; break;
    case MOE_BWS_DY_LATENT: o = B.dyr; n = cfg->d_latent ? t * cfg->d_latent * 2 : 0; break;
    default: return MOE_ERR_INVALID_ARG;
  }
  *offset = o;
  *bytes = n;
  return MOE_OK;
}

moe_status_t moe_layer_backward(const moe_config_t* cfg, int32_t T, const void* x, const moe_weights_t* w,
                                const void* dy, const int32_t* topk_ids, const float* topk_w, const float* scores,
                                float* dx, const moe_grads_t* grads, const void* ws, size_t ws_bytes, void* bws,
                                size_t bws_bytes, void* stream) {
  moe_status_t st = check_backward(cfg, T, ws, ws_bytes, bws, bws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, true, true)) != MOE_OK) return st;
  if (!grads) return MOE_ERR_INVALID_ARG;
  REQ(x); REQ(dy); REQ(topk_ids); REQ(topk_w); REQ(scores); REQ(dx);
  OPT(grads->d_router); OPT(grads->d_lat_down); OPT(grads->d_lat_up); OPT(grads->d_up); OPT(grads->d_down);
  OPT(grads->d_sh_up); OPT(grads->d_sh_down);
  Ptrs P{(char*)const_cast<void*>(ws), make_layout(cfg, T)};
  return run_backward(cfg, T, x, w, dy, topk_ids, topk_w, scores, dx, grads, P, (char*)bws, (cudaStream_t)stream);
}

moe_status_t moe_block_backward(const moe_config_t* cfg, int32_t T, const void* x, const float* norm_w,
                                float norm_eps, const void* x_norm, const moe_weights_t* w, const void* dout,
                                const int32_t* topk_ids,
                                const float* topk_w, const float* scores, float* dx, const moe_grads_t* grads,
                                const void* ws, size_t ws_bytes, void* bws, size_t bws_bytes, void* stream) {
  moe_status_t st = check_backward(cfg, T, ws, ws_bytes, bws, bws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_weights(cfg, w, true, true, true)) != MOE_OK) return st;
  if (!grads) return MOE_ERR_INVALID_ARG;
  REQ(x); REQ(norm_w); REQ(dout); REQ(topk_ids); REQ(topk_w); REQ(scores); REQ(dx); OPT(x_norm);
  OPT(grads->d_norm_w);
  if (!std::isfinite(norm_eps) || norm_eps < 0.f) return MOE_ERR_INVALID_ARG;
  Ptrs P{(char*)const_cast<void*>(ws), make_layout(cfg, T)};
  const BwLayout B = make_bw_layout(cfg, T);
  char* b = (char*)bws;
  cudaStream_t s = (cudaStream_t)stream;
  float* dxn = reinterpret_cast<float*>(b + B.dxn);
  // the layer read the normalised rows the block's forward wrote (x_norm_out, or the workspace)
  const void* xn = x_norm ? x_norm : P.at<void>(P.L.xn);
  if ((st = run_backward(cfg, T, xn, w, dout, topk_ids, topk_w, scores, dxn, grads, P, b, s)) != MOE_OK) return st;
  CU(launch_rmsnorm_bwd(x, norm_w, norm_eps, T, cfg->d_model, dout, dxn, dx, reinterpret_cast<float*>(b + B.xr),
                        grads->d_norm_w, s));
  return MOE_OK;
}

moe_status_t moe_get_device_error(const void* ws, void* stream, int32_t* code) {
  if (!ws || !code) return MOE_ERR_INVALID_ARG;
  int32_t v = 0;
  CU(cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream));
  CU(cudaStreamSynchronize((cudaStream_t)stream));
  *code = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status_t moe_clear_device_error(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  CU(cudaMemsetAsync(ws, 0, sizeof(int32_t), (cudaStream_t)stream));
  return MOE_OK;
}

moe_status_t moe_layer_forward_host(const moe_config_t* cfg, int32_t T, const void* x_host, void* x_dev,
                                    const moe_weights_t* w, void* y_dev, void* y_host, void* ws, size_t ws_bytes,
                                    void* stream) {
  moe_status_t st = check_common(cfg, T, ws, ws_bytes);
  if (st != MOE_OK || T == 0) return st;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  REQ(x_dev); REQ(y_dev);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = (size_t)T * cfg->d_model * act_bytes(cfg);
  CU(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s));
  st = moe_layer_forward(cfg, T, x_dev, w, y_dev, nullptr, nullptr, nullptr, nullptr, ws, ws_bytes, stream);
  if (st != MOE_OK) return st;
  CU(cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, s));
  CU(cudaStreamSynchronize(s));
  return MOE_OK;
}

}  // extern "C"
