// Internal launchers shared between the translation units of the library.
#pragma once

#include "common.cuh"

#include <mutex>

namespace moe {

// host-side count of kernel launches (moe_launch_count)
void count_launches(int n);

// One-time set-up that belongs to a device (a kernel's shared-memory limit set
// by cudaFuncSetAttribute, a resident-CTA count): run once per device index,
// with that device current, and the result kept per device, so a process that
// drives several GPUs sets each one up.  Thread-safe.
constexpr int kMaxDevices = 64;
struct PerDeviceOnce {
  std::once_flag flag[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
  int val[kMaxDevices] = {};
  // fn(int& value) -> cudaError_t runs on the first call for the current
  // device; *value receives the value it stored
  template <class F>
  cudaError_t run(F&& fn, int* value = nullptr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { err[dev] = fn(val[dev]); });
    if (value) *value = val[dev];
    return err[dev];
  }
};

// Launch with programmatic stream serialisation (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// epilogues of the streaming GEMV / grouped GEMM kernels
enum Epi : int {
  EPI_RELU2 = 0,  // out = bf16(relu(bf16(v))^2)            (F32 layers: relu(v)^2)
  EPI_SCALE = 1,  // out(f32) = topk_w[route] * v            (expert down: routed row u)
  EPI_STORE = 2,  // out = bf16(v)                           (F32 out: v)
  EPI_ADD = 3     // out = bf16(v + add_src[row, f] + res[row, f])   (F32 out: no rounding)
};

// Weight formats of the streamed matrix
enum WFmt : int { WF_BF16 = 0, WF_F32 = 1, WF_NVFP4 = 2 };

// One "grouped" matrix-times-rows product: for every segment (an active
// expert, or one dense segment) out[rows, N] = X[rows, K] W_seg[N, K]^T.
struct GemvArgs {
  const void* W;            // [segments][N][K] (NVFP4: packed bytes [segments][N][K/2])
  const uint8_t* W_sf;      // NVFP4 block scales [segments][N][K/16]
  const float* W_gs;        // NVFP4 per-tensor scales [segments]
  int64_t w_seg_stride;     // elements (bytes for NVFP4) between segments
  int64_t sf_seg_stride;    // bytes between segments' scales
  int N, K;
  const void* X;            // activation rows, row stride x_ld elements
  int64_t x_ld;
  const int32_t* gather;    // X row of logical row r (route_token) or nullptr
  const int32_t* offsets;   // [E+1] segment rows (grouped) or nullptr (dense)
  const int32_t* active;    // [E] active expert list (grouped)
  const WsHeader* hdr;      // n_active (grouped)
  int dense_rows;           // rows of the dense segment
  void* out;                // out rows [rows, out_ld]
  int64_t out_ld;
  const float* add_src;     // EPI_ADD source [rows, add_ld] f32 (nullable: adds 0)
  int64_t add_ld;
  // EPI_ADD residual [rows, res_ld] in the activation type (nullable), added
  // after add_src, before the one rounding; an output row may be its own
  // residual row (each element is read before it is written, by one thread)
  const void* res;
  int64_t res_ld;
  const float* topw;        // EPI_SCALE: [T, K] routing weights
  const int32_t* route_token;
  const int32_t* route_slot;
  int top_k;
  int32_t* err;
  // NVFP4 streaming GEMV only (gemv_nvfp4_streams): X holds FP16 activations
  // (the exact FP16 copy of BF16 ones); out receives FP16 copies of the
  // BF16-rounded outputs
  bool x_f16, out_f16;
  // FP4 tensor-core products only (launch_gemm_fp4): X holds the rows' NVFP4
  // activation terms [x_terms][x_rows_cap][K/2] bytes, X_sf their E4M3 block
  // scales [x_terms][x_rows_cap][x_sf_ld] bytes, x_scale the rows' FP32 scale
  const uint8_t* X_sf;
  int64_t x_sf_ld;
  const float* x_scale;
  int64_t x_rows_cap;
  int x_terms;
};

// act: MOE_DT_BF16 / MOE_DT_F32 activation type of X and of non-f32 outputs.
// out_f32: output element type is f32 (else act type).
cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int act, int epi, bool out_f32,
                        int max_rows, int grid_segments, cudaStream_t s);

// true when launch_gemv runs a grouped NVFP4 product (BF16 activations) with
// the streaming kernel, the one that accepts x_f16 / out_f16
bool gemv_nvfp4_streams(const GemvArgs& a);

// out[i] = FP16(x[i]) for n BF16 values (n a multiple of 8, 16-byte aligned)
// (err: MOE_DEVERR_RANGE is set there when a value is beyond FP16's range)
cudaError_t launch_bf16_to_f16(const void* x, int64_t n, void* out, cudaStream_t s, int32_t* err);

// Tensor-core grouped GEMM (tcgen05): same arguments as launch_gemv; X rows must
// be contiguous (no gather).  w_rows/x_rows: rows of the W and X matrices (TMA
// extents); E: segments (0 = dense); bn: rows per tile (power of two, 16..256).
// x_cols < K (a divisor of K) re-reads X's first x_cols columns for every
// x_cols-wide slice of W's K (used to multiply X by side-by-side split parts of
// one matrix); 0 = K.
// ksplit > 1 (dense FP32 stores only) splits K into that many parts, each a
// separate output slab [x_rows, out_ld] after the previous one; the caller adds
// the slabs in part order.
cudaError_t launch_gemm_tc(const GemvArgs& a, int epi, bool out_f32, int64_t w_rows, int64_t x_rows, int E, int bn,
                           cudaStream_t s, int x_cols = 0, int ksplit = 1);
// Rows per tile for launch_gemm_tc: the largest power of two (16..256) that
// still gives every SM about two tiles, for segments of rows_per_seg rows and
// N output features.
int tc_tile_rows(int64_t rows_per_seg, int64_t segs, int N);

// NVFP4 activation terms and the FP4 tensor-core grouped GEMM (gemm_fp4.cu).
// A row of K activations becomes kActTerms NVFP4 terms (residual
// quantisation: each term encodes what the earlier ones left), so both
// operands of an expert product are NVFP4 and the block-scaled FP4 MMA
// multiplies them; the term count trades accuracy (about 0.18^n of a 16-value
// block's largest magnitude left over) for MMA work.
constexpr int kActTerms = 3;
constexpr int kActTermsMax = 4;
// row stride of a term's block scales (K/16 bytes rounded up to 16 for TMA)
inline int64_t act_sf_ld(int K) { return ((int64_t)K / 16 + 15) / 16 * 16; }
// rows r < (*count if count else R) of x (BF16, row stride x_ld elements;
// row r reads x[gather[r]] when gather is given) -> terms q [nterms][rows_cap]
// [K/2], scales sf [nterms][rows_cap][act_sf_ld(K)], row scale g [rows_cap]
cudaError_t launch_quant_terms(const void* x, int64_t x_ld, const int32_t* gather, const int32_t* count, int R, int K,
                               int nterms, uint8_t* q, uint8_t* sf, float* g, int64_t rows_cap, cudaStream_t s);
// out = epilogue(W_seg x_terms) for grouped (a.offsets) or dense products;
// a.W / a.W_sf / a.W_gs: NVFP4 weights [w_rows, K/2] u8, E4M3 scales
// [w_rows, K/16], per-segment FP32 scales; a.X / a.X_sf / a.x_scale: the
// activation terms above.  bn: rows per tile (16..128, a multiple of 16).
cudaError_t launch_gemm_fp4(const GemvArgs& a, int epi, bool out_f32, int64_t w_rows, int E, int bn, cudaStream_t s);
int fp4_tile_rows(int64_t rows_per_seg, int64_t segs, int N);

// router
// w_split: scratch of E * 3d BF16 for the tensor-core path (many BF16 tokens);
// nullptr keeps the FP32 SIMT kernels.  parts: scratch of kRouterParts * T * E
// FP32 for K-split tensor-core logits (nullptr: no split).  *nparts receives
// the number of logit slabs written (1: `logits` itself; more: `parts`, slab p
// at p * T * E), which the selection kernel adds in order.
constexpr int kRouterParts = 4;
cudaError_t launch_router_logits(const void* x, int act, int T, int d, const float* w_router, int E,
                                 float* logits, cudaStream_t s, void* w_split, float* parts, int* nparts);
// logits: slab 0 of nparts slabs part_stride floats apart; their sum (part
// order) is the logit, written to logits_out when it is not nullptr
cudaError_t launch_router_select(const float* logits, int nparts, int64_t part_stride, float* logits_out, int T,
                                 int E, const float* bias, int G, int TG, int K, int norm, float rsf, float* scores,
                                 int32_t* ids, float* w, int32_t* err, cudaStream_t s);

// dispatch
struct DispatchArgs {
  const int32_t* ids;
  int T, K, E;
  int32_t* counts;
  int32_t* offsets;
  int32_t* route_token;
  int32_t* route_slot;
  int32_t* token_slot_row;
  int32_t* active;          // [E]
  WsHeader* hdr;
  int32_t* tile_counts;     // [n_tiles, E] (multi-CTA path)
  int32_t* tile_prefix;     // [E+1] tensor-core tile prefix (nullable)
  int tile_rows;            // rows per tensor-core tile (0 = no tile prefix)
  const void* x_e;          // pack source [T, de] (nullable)
  void* x_packed;           // pack destination [R, de] (nullable)
  int de;
  int elem_bytes;
  bool pack_f16;            // BF16 rows packed as their FP16 copies
};
size_t dispatch_tile_count_elems(int T, int K, int E);
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s);
// x_packed[j] = x_e[route_token[j]] for the offsets[E] <= R packed rows (rows
// of de elements of elem_bytes; to_f16: BF16 rows stored as FP16 copies)
cudaError_t launch_pack_rows(const void* x_e, const int32_t* route_token, const int32_t* offsets, int E, int R,
                             int de, int elem_bytes, bool to_f16, void* x_packed, cudaStream_t s,
                             int32_t* err = nullptr);

// selection arguments (see launch_router_select)
struct SelectArgs {
  const float* logits;
  int nparts;
  int64_t part_stride;
  float* logits_out;
  int T, E;
  const float* bias;
  int G, TG, K, norm;
  float rsf;
  float* scores;
  int32_t* ids;
  float* w;
  int32_t* err;
};
// Selection followed by dispatch in one single-CTA kernel, for a few tokens
// (T <= 16, T*K <= 256) on the GEMV path (no tile schedule, no packed rows);
// same results as launch_router_select + launch_dispatch.
bool select_dispatch_fits(int T, int K, const DispatchArgs& a);
cudaError_t launch_select_dispatch(const SelectArgs& sa, const DispatchArgs& a, cudaStream_t s);

// combine: y_r[t] = sum over t's packed rows in ascending order of u[row];
// y_r_act[t] = act(y_r[t] + add[t] + res[t]) (add: f32, res: act dtype, both
// nullable; y_r_act may be res itself)
cudaError_t launch_combine(const float* u, const int32_t* token_slot_row, int T, int K, int de,
                           float* y_r, void* y_r_act, int act, cudaStream_t s, const float* add = nullptr,
                           const void* res = nullptr);

// dst (act dtype) = act(src (f32) + res (act dtype, nullable)), n a multiple of 4
cudaError_t launch_cast(const float* src, int64_t n, void* dst, int act, cudaStream_t s, const void* res = nullptr);

// ReLU^2-sparse down projection (decode): W in the group-major layout of
// moe_sparse_down_layout, X = h (BF16, or FP16 with NVFP4 weights), grouped
// rows (offsets / active / hdr), EPI_SCALE output; only the 16-neuron groups
// with a nonzero h value in one of an expert's rows are read
bool sparse_down_fits(int N, int K, bool nvfp4);
cudaError_t launch_sparse_down(const GemvArgs& a, bool nvfp4, int segs, cudaStream_t s);
cudaError_t launch_sparse_down_layout(const void* w, const uint8_t* sf, int E, int de, int I, bool nvfp4, void* out,
                                      void* out_sf, cudaStream_t s);

// ---- backward -------------------------------------------------------------
// Grouped BF16 GEMM of the backward, C[m, n] = sum_k A[m, k] B[k, n], FP32
// accumulation.  GM_ROWS: the rows of expert segment e (offsets / active /
// hdr, or dense_rows rows when offsets is NULL) times B + e * b_seg (K = K);
// GM_KSEG: C + e * c_seg [M, N] from K = the segment's rows.  A is [m][k]
// (a_t = false; a_gather maps m to an A row) or [k][m] (a_t = true); B is
// [k][n] (b_gather maps k to a B row).  Dimensions: N % 8 == 0; GM_ROWS:
// K % 32 == 0; GM_KSEG: M % 8 == 0.
enum { GM_ROWS = 0, GM_KSEG = 1 };
enum {
  GE_ACC_F32 = 0,      // C (f32) += acc
  GE_STORE_F32 = 1,    // C (f32) = acc
  GE_STORE_BF16 = 2,   // C (bf16) = bf16(acc)
  GE_RELU2_GRAD = 3    // C (bf16) = bf16(acc * 2 sqrt(aux)), aux: BF16 h = relu(a)^2 at [m][n]
};
struct GemmArgs {
  int mode, epi;
  const bf16* A;
  int64_t lda;
  bool a_t;
  const int32_t* a_gather;
  const bf16* B;
  int64_t ldb, b_seg;
  const int32_t* b_gather;
  void* C;
  int64_t ldc, c_seg;
  int M, N, K;
  const int32_t* offsets;
  const int32_t* active;
  const WsHeader* hdr;
  int dense_rows;
  const bf16* aux;
  int64_t aux_ld;
  const int32_t* tprefix;   // GM_ROWS over segments: 64-row tile prefix (launch_tile_scan)
};
// segs: active segments launched (1 for a dense product); rows: all rows
// (GM_ROWS: the sum over segments, or the dense rows)
cudaError_t launch_gemm_bwd(const GemmArgs& g, int segs, int rows, cudaStream_t s);
cudaError_t launch_tile_scan(const int32_t* offsets, const int32_t* active, const WsHeader* hdr, int32_t* tprefix,
                             cudaStream_t s);
// combine backward: packed row r = (t, k): dU[r] = bf16(w_tk dy[t]), q[t, k] = <dy[t], u[r]> / w_tk
cudaError_t launch_combine_bwd(const void* dy, int64_t dy_ld, const float* u, const int32_t* rt, const int32_t* rs,
                               const float* topw, int R, int K, int de, void* dU, float* q, cudaStream_t s);
// gate backward: dz[t, k] from q and the chosen scores
cudaError_t launch_gate_bwd(const float* scores, const int32_t* ids, const float* q, int T, int E, int K, int norm,
                            float rsf, float* dz, cudaStream_t s);
// dW_r[e] += sum over expert e's packed rows of dz x[token]
cudaError_t launch_router_wgrad(const void* x, bool x_f32, int d, const float* dz, const int32_t* rt,
                                const int32_t* rs, int K, const int32_t* offsets, const int32_t* active,
                                const WsHeader* hdr, int segs, float* dW, cudaStream_t s);
// dx[t] = sum_k dz_tk W_r[id_tk] + a[t] + b[t]
cudaError_t launch_input_grad(const float* dz, const int32_t* ids, int T, int K, const float* w_router, int d,
                              const float* a, const float* b, float* dx, cudaStream_t s);
// RMSNorm backward of the block (BF16 x and dout): dx, and dgamma += (if not NULL)
cudaError_t launch_rmsnorm_bwd(const void* x, const float* gamma, float eps, int T, int d, const void* dout,
                               const float* dxn, float* dx, float* xr, float* dgamma, cudaStream_t s);

// RMSNorm prologue of a block: xn[t] = act(gamma * (x[t] / sqrt(mean(x[t]^2) + eps)))
// in FP32 (x, xn: act dtype [T, d]; gamma: f32 [d]); block 0 also clears the
// workspace header `hdr` (bytes), so that it replaces the step's header memset
cudaError_t launch_rmsnorm(const void* x, const float* gamma, float eps, int T, int d, int act, void* xn,
                           void* hdr, int hdr_bytes, cudaStream_t s);

}  // namespace moe
