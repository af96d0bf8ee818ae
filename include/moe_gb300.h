/*
 * moe_gb300.h -- C ABI of the routed ReLU^2 mixture-of-experts layer
 * (NemotronH-style MoE feed-forward block), hand-written CUDA for sm_103a.
 *
 * The layer, for hidden rows x[T, d]:
 *   (latent shapes)  x_e = bf16(x W_ld^T)                       [T, L]      else x_e = x
 *   router           z = x W_r^T (FP32), s = sigmoid(z) (FP32),
 *                    group-limited top-K on c = s + b, weights from s,
 *                    normalised, times routed_scaling_factor
 *   dispatch         per-expert counts, exclusive scan, routes sorted by
 *                    (expert, token, slot)
 *   experts          h = bf16(relu(bf16(x_e W_up,e^T))^2);  u = w * (h W_down,e^T)  (FP32)
 *   combine          y_r[t] = sum of t's routed rows in ascending expert id (FP32)
 *   shared + output  y_s = W_sd bf16(relu(bf16(W_su x))^2)  (FP32)
 *                    y = bf16(y_r + y_s)                       (no latent)
 *                    y = bf16(bf16(y_r) W_lu^T + y_s)          (latent)
 * Sources: page "Nemotron Is Not One Circuit: Mamba, Attention, and MoE
 * Routing" (sections "The Four Layer Kinds CKE Must Preserve", "The Router Is
 * A Deterministic Algorithm", "The C Kernel Contract"); page "M6.1 - Routed
 * Capacity: MoE Experts, Routers, and Token Dispatch" (sections 0x04A,
 * 0x05A-0x05F); page "NemotronH (Nemotron 3.5 Lightning, Bolt, Super VL)"
 * (section "Arithmetic"); page "Nemotron-3.5-Super 120B on an 8 GB GPU"
 * (section "The only number that matters", latent experts; section "The
 * engine, step by step", item 4, NVFP4 block scales).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise, allocated and owned
 *    by the caller; the library never allocates device memory, frees or
 *    synchronises (except moe_get_device_error and the _host convenience
 *    call).  Every call only enqueues work on `stream` (a cudaStream_t passed
 *    as void*; NULL = the legacy default stream) and returns.
 *    moe_layer_forward (and moe_block_forward) runs the latent down
 *    projection and the shared expert on a library-owned auxiliary stream
 *    (one per device, created with its events on the first call), forked
 *    from and joined back to `stream` by events, so the layer is still
 *    ordered as one operation on `stream`.  Calls from several host threads
 *    take turns enqueuing (a per-device lock is held while a call enqueues),
 *    and their auxiliary work runs one call after another on that one
 *    stream: correct, but two layers on different caller streams overlap
 *    only in their routed parts.
 *  - Row-major storage.  Weight matrices are stored [out, in] (the
 *    nn.Linear orientation, page "M6.1 ...", section 0x04A).
 *  - Every device pointer must be 16-byte aligned; every inner width
 *    (d_model, d_latent, d_expert, d_shared) a multiple of 64.
 *  - Argument and shape errors are returned before anything is enqueued.
 *    A failed launch returns MOE_ERR_CUDA.  Conditions only the device can see
 *    (an expert id out of range, a non-finite router score) set bits of the
 *    device error word held in the workspace; read it with
 *    moe_get_device_error.  Kernels never trap or assert.
 *  - Outputs are overwritten, never accumulated into.
 *  - Results are bit-identical from run to run for the same inputs and T
 *    (no floating-point atomics; every sum has a fixed order).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status_t;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape or parameter */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not built (e.g. a width not a multiple of 64) */
  MOE_ERR_WORKSPACE = 3,    /* workspace smaller than moe_workspace_bytes() */
  MOE_ERR_CUDA = 4,         /* a CUDA call or launch failed */
  MOE_ERR_DEVICE = 5        /* moe_get_device_error found a device-side error bit */
};

/* device error word bits (moe_get_device_error) */
enum {
  MOE_DEVERR_EXPERT_ID = 1,      /* an expert id outside [0, n_experts) reached dispatch */
  MOE_DEVERR_NONFINITE = 2,      /* a router score was NaN (ranked last, never chosen before a finite one) */
  MOE_DEVERR_SCHEDULE = 4,       /* a tile schedule disagreed with the dispatch offsets */
  MOE_DEVERR_TIMEOUT = 8,        /* a kernel's bounded wait expired; that kernel stopped early */
  MOE_DEVERR_RANGE = 16          /* NVFP4 experts on the FP16 path (under 8 tokens, or above 64): a value
                                    beyond FP16's range (|v| > 65504) reached an FP16 operand (expert
                                    input row or h); the affected outputs are not finite.  The FP4
                                    tensor path (8..64 tokens) carries each row's magnitude in its
                                    FP32 row scale and has no such limit */
};

typedef int32_t moe_dtype_t;
enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1, MOE_DT_NVFP4 = 2 };

typedef struct moe_config {
  int32_t d_model;       /* d: hidden width */
  int32_t d_latent;      /* L: latent width the experts act on; 0 = experts act on d */
  int32_t n_experts;     /* E: routed experts, 1..1024 */
  int32_t top_k;         /* K: experts per token, 1..min(E, 32) */
  int32_t n_group;       /* G: equal contiguous expert groups (E % G == 0) */
  int32_t topk_group;    /* TG: groups kept per token, 1..G */
  int32_t d_expert;      /* I: routed expert intermediate width */
  int32_t d_shared;      /* S: shared expert intermediate width; 0 = no shared expert */
  int32_t norm_topk_prob;          /* 1: chosen weights normalised to sum 1 before scaling */
  float routed_scaling_factor;     /* multiplies the (normalised) chosen weights */
  moe_dtype_t act_dtype;           /* MOE_DT_BF16 or MOE_DT_F32 (activations, dense weights) */
  moe_dtype_t expert_dtype;        /* MOE_DT_BF16, MOE_DT_F32 (with F32 activations) or MOE_DT_NVFP4 */
} moe_config_t;

/* Weights of one layer (device pointers, row-major [out, in]).  de = L if L>0 else d.
 * Dense tensors use act_dtype; routed experts use expert_dtype.               */
typedef struct moe_weights {
  const float* w_router;      /* [E, d]  FP32 router matrix                                  */
  const float* router_bias;   /* [E]     FP32 selection bias, or NULL (choice only)          */
  const void* w_lat_down;     /* [L, d]  latent down (latent shapes only)                    */
  const void* w_lat_up;       /* [d, L]  latent up   (latent shapes only)                    */
  const void* w_up;           /* [E, I, de] expert up   (BF16/F32) or NVFP4 packed [E, I, de/2] u8   */
  const void* w_down;         /* [E, de, I] expert down (BF16/F32) or NVFP4 packed [E, de, I/2] u8   */
  const uint8_t* w_up_sf;     /* NVFP4: E4M3 block scales [E, I, de/16], one per 16 K-elements       */
  const uint8_t* w_down_sf;   /* NVFP4: E4M3 block scales [E, de, I/16]                              */
  const float* w_up_gs;       /* NVFP4: FP32 per-tensor scale [E]                                    */
  const float* w_down_gs;     /* NVFP4: FP32 per-tensor scale [E]                                    */
  const void* w_sh_up;        /* [S, d] shared expert up   (S > 0)                                    */
  const void* w_sh_down;      /* [d, S] shared expert down (S > 0)                                    */
  /* optional: the expert down weights again, in the group-major layout of
   * moe_sparse_down_layout (NULL = not given).  When given, decode steps of
   * up to 16 tokens (BF16 experts; NVFP4 experts on their FP16 path)
   * compute the down projection by the ReLU^2-sparse kernel, which reads
   * only the 16-neuron groups of W_down with a live neuron.                 */
  const void* w_down_g;       /* BF16 [E, de * I] / NVFP4 values [E, de * I / 2] u8                   */
  const uint8_t* w_down_g_sf; /* NVFP4: E4M3 scales [E, de * I / 16]                                  */
} moe_weights_t;

/* Library version, e.g. 100 for 0.1.0.  Never fails. */
int32_t moe_version(void);

/* Short static description of a status code.  Never fails. */
const char* moe_status_string(moe_status_t s);

/* Validates a configuration without touching any pointer. */
moe_status_t moe_check_config(const moe_config_t* cfg);

/* Bytes of device workspace moe_layer_forward needs for T tokens (0 on an
 * invalid configuration).  The same workspace serves every step entry point;
 * its first 256 bytes hold the device error word and the expert schedule that
 * moe_dispatch leaves for moe_experts_up / moe_experts_down_combine.  The
 * error word is sticky: clear it once on a new workspace (zero the first 256
 * bytes, or moe_clear_device_error) before reading it. */
size_t moe_workspace_bytes(const moe_config_t* cfg, int32_t T);

/* Step 1: router (page "Nemotron Is Not One Circuit", sections "The Router Is
 * A Deterministic Algorithm" and "The C Kernel Contract"; page "NemotronH ...",
 * section "Arithmetic", router bullet).
 *   x        [T, d] act_dtype hidden rows (BF16 values enter FP32 exactly)
 *   logits   [T, E] FP32 out: z = x W_r^T, or NULL (kept in the workspace)
 *   scores   [T, E] FP32 out: s = sigmoid(z), or NULL
 *   topk_ids [T, K] int32 out: chosen experts, best biased score first,
 *            equal scores to the lower id
 *   topk_w   [T, K] FP32 out: s of the chosen experts, normalised (if
 *            configured) then times routed_scaling_factor                   */
moe_status_t moe_router(const moe_config_t* cfg, int32_t T, const void* x,
                        const float* w_router, const float* router_bias,
                        float* logits, float* scores, int32_t* topk_ids, float* topk_w,
                        void* ws, size_t ws_bytes, void* stream);

/* Step 2: dispatch (page "M6.1 ...", sections 0x05A "The Route Row Is The
 * Reversible Unit" and 0x05B).  Routes r = (token t, slot k) are laid out
 * expert-contiguously, sorted by (expert, token, slot); no atomics.
 *   topk_ids       [T, K] int32 in
 *   x_e            [T, de] act_dtype rows to pack (x, or the latent rows), or NULL
 *   counts         [E] int32 out: routes per expert
 *   offsets        [E+1] int32 out: exclusive prefix sum of counts
 *   route_token    [T*K] int32 out: token of each packed row
 *   route_slot     [T*K] int32 out: slot of each packed row
 *   token_slot_row [T, K] int32 out: packed row of route (t, k)
 *   x_packed       [T*K, de] out: x_packed[j] = x_e[route_token[j]], or NULL
 * Also leaves the expert schedule in the workspace header.                   */
moe_status_t moe_dispatch(const moe_config_t* cfg, int32_t T, const int32_t* topk_ids,
                          const void* x_e, int32_t* counts, int32_t* offsets,
                          int32_t* route_token, int32_t* route_slot, int32_t* token_slot_row,
                          void* x_packed, void* ws, size_t ws_bytes, void* stream);

/* Step 3: expert up projections with squared ReLU, no gate (page "NemotronH
 * ...", section "Arithmetic": bf16(relu(bf16(up x))^2)).
 *   x_e         [T, de] rows the experts read (gathered through route_token),
 *               ignored when x_packed is given
 *   x_packed    [T*K, de] packed rows from moe_dispatch, or NULL (above 64
 *               BF16 tokens, where the tensor-core kernel reads contiguous
 *               rows, x_e is then first gathered into the workspace)
 *   route_token, offsets: from moe_dispatch (same workspace)
 *   h           [T*K, I] out, packed order; BF16 (F32 for F32 layers)        */
moe_status_t moe_experts_up(const moe_config_t* cfg, int32_t T, const void* x_e,
                            const void* x_packed, const int32_t* route_token,
                            const int32_t* offsets, const moe_weights_t* w, void* h,
                            void* ws, size_t ws_bytes, void* stream);

/* Steps 4+5: expert down projections, times the routing weight, and the
 * combine: y_routed[t] = sum over t's routes in ascending expert id of
 * w_tk * (h_r W_down,e^T), all FP32 (page "NemotronH ...", section
 * "Arithmetic"; page "M6.1 ...", section 0x05B, weighted scatter-add).
 *   h              [T*K, I] from moe_experts_up
 *   route_token, route_slot, token_slot_row, offsets: from moe_dispatch
 *   topk_w         [T, K] FP32 from moe_router
 *   y_routed       [T, de] FP32 out                                         */
moe_status_t moe_experts_down_combine(const moe_config_t* cfg, int32_t T, const void* h,
                                      const int32_t* offsets, const int32_t* route_token,
                                      const int32_t* route_slot, const int32_t* token_slot_row,
                                      const float* topk_w, const moe_weights_t* w,
                                      float* y_routed, void* ws, size_t ws_bytes, void* stream);

/* Step 4 alone: the expert down projections times the routing weights, one
 * FP32 row per route in packed order, without the combine (page "NemotronH
 * ...", section "Arithmetic": the down projection accumulates in FP32; page
 * "M6.1 ...", section 0x05B, the gate-weighted routed rows).
 *   h, offsets, route_token, route_slot, topk_w: as for moe_experts_down_combine
 *   u   [T*K, de] FP32 out: u[r] = topk_w[t, k] * (h_r W_down,e^T) for packed
 *       row r of route (t, k) to expert e                                    */
moe_status_t moe_experts_down(const moe_config_t* cfg, int32_t T, const void* h, const int32_t* offsets,
                              const int32_t* route_token, const int32_t* route_slot, const float* topk_w,
                              const moe_weights_t* w, float* u, void* ws, size_t ws_bytes, void* stream);

/* Latent down projection of latent shapes: x_l = bf16(x W_ld^T), FP32
 * accumulation (page "Nemotron-3.5-Super 120B on an 8 GB GPU", section "The
 * only number that matters": experts work in a 1024-wide latent space).
 *   x [T, d] in, x_l [T, L] out (act_dtype).                                  */
moe_status_t moe_latent_down(const moe_config_t* cfg, int32_t T, const void* x,
                             const moe_weights_t* w, void* x_l,
                             void* ws, size_t ws_bytes, void* stream);

/* Shared expert and output (page "Nemotron Is Not One Circuit", section "The
 * Four Layer Kinds CKE Must Preserve": routed experts + shared expert).
 *   x        [T, d] hidden rows
 *   y_routed [T, de] FP32 combined routed output, or NULL (treated as zero)
 *   y        [T, d] act_dtype out: bf16(y_routed + y_s), or for latent shapes
 *            bf16(bf16(y_routed) W_lu^T + y_s); y_s = 0 when S == 0        */
moe_status_t moe_shared(const moe_config_t* cfg, int32_t T, const void* x,
                        const moe_weights_t* w, const float* y_routed, void* y,
                        void* ws, size_t ws_bytes, void* stream);

/* The whole layer, every step above on `stream`, intermediates in `ws`.
 *   x [T, d] in; y [T, d] out (act_dtype).
 *   topk_ids_out [T,K] / topk_w_out [T,K] / logits_out [T,E] / scores_out [T,E]:
 *   optional copies of the router's results (NULL = not written).
 * Clears the device error word first.  NVFP4 experts: see
 * moe_set_nvfp4_act_terms for how the activations enter their products.     */
moe_status_t moe_layer_forward(const moe_config_t* cfg, int32_t T, const void* x,
                               const moe_weights_t* w, void* y,
                               int32_t* topk_ids_out, float* topk_w_out,
                               float* logits_out, float* scores_out,
                               void* ws, size_t ws_bytes, void* stream);

/* ReLU^2-sparse down projection for decode (page "Nemotron-3.5-Super 120B on
 * an 8 GB GPU", section "The engine, step by step", item 4 "Skip the zeros",
 * and section "What didn't work": 16-neuron groups, not single neurons).
 * The down weights are re-laid once, a pure permutation of their values (and,
 * NVFP4, of their bytes and scales), so that each group of 16 neurons
 * 16g .. 16g+15 of an expert holds all de outputs' weights for those neurons
 * contiguously.  Within a group, 16-output tile o is one 512-byte block
 * (BF16) in which lane l = 4r + t (r = l / 4, t = l % 4) holds 16 bytes:
 * W[16o + r][16g + 4t .. +3] then W[16o + r + 8][16g + 4t .. +3].  NVFP4:
 * 64-output quad q of a group is one 512-byte value block, lane l holding
 * for tiles j = 0..3 of the quad the 2 bytes of W[64q + 16j + r][16g + 4t ..
 * +3] then the 2 bytes of row + 8 (low nibble = even neuron, as in w_down),
 * and one 64-byte scale block, bytes 8r + 2j and 8r + 2j + 1 holding the
 * group's E4M3 scales of rows 64q + 16j + r and 64q + 16j + r + 8.
 * A decode step that is given w_down_g finds, per expert, the groups with a
 * nonzero h value in any of the expert's rows and reads only those groups'
 * weights; dead groups only contribute zeros, so the result is that of the
 * dense product up to the order of its FP32 sum.  Needs BF16 activations,
 * I % 16 == 0, I / 16 <= 1024 and de % 32 == 0 (BF16) or de % 64 == 0
 * (NVFP4); else MOE_ERR_UNSUPPORTED.
 * moe_sparse_down_bytes: sizes of w_down_g (*values) and w_down_g_sf
 * (*scales, 0 for BF16).  moe_sparse_down_layout: writes both from w->w_down
 * (and w->w_down_sf) on `stream` (caller-owned, 16-byte aligned buffers).  */
moe_status_t moe_sparse_down_bytes(const moe_config_t* cfg, size_t* values, size_t* scales);
moe_status_t moe_sparse_down_layout(const moe_config_t* cfg, const moe_weights_t* w, void* w_down_g,
                                    uint8_t* w_down_g_sf, void* stream);

/* The MoE block of a decoder layer: RMSNorm, the layer, the residual add
 * (page "Nemotron Is Not One Circuit: Mamba, Attention, and MoE Routing",
 * section "The Four Layer Kinds CKE Must Preserve": an MoE layer is RMSNorm,
 * router, group-limited top-k, routed ReLU^2 experts + shared expert,
 * residual).  Chains of blocks need no host work between them, so several
 * can be captured in one CUDA graph (page "NemotronH (Nemotron 3.5 Lightning,
 * Bolt, Super VL)", section "Speculation": verify blocks of 1-16 rows).
 *   x        [T, d] act_dtype residual stream in
 *   norm_w   [d] FP32 RMSNorm weight gamma;  norm_eps >= 0
 *   out      [T, d] act_dtype: out = act(x + layer(xn)), the layer's FP32
 *            output and the residual added before the one rounding.  out may
 *            be x itself (in place); any other overlap with x is rejected.
 *   xn = act(gamma * (x * r)), r = 1 / sqrt(mean(x^2) + eps) per row, all in
 *            FP32 with one rounding: the rows the router, the latent down
 *            projection, the shared expert and (without a latent) the experts
 *            read.  x_norm_out [T, d]: an optional copy (NULL: kept in the
 *            workspace, MOE_WS_X_NORM); it must not overlap x or out.
 *   topk_ids_out / topk_w_out / logits_out / scores_out: as moe_layer_forward.
 * The RMSNorm kernel also clears the workspace header (no separate memset). */
moe_status_t moe_block_forward(const moe_config_t* cfg, int32_t T, const void* x,
                               const float* norm_w, float norm_eps,
                               const moe_weights_t* w, void* out, void* x_norm_out,
                               int32_t* topk_ids_out, float* topk_w_out,
                               float* logits_out, float* scores_out,
                               void* ws, size_t ws_bytes, void* stream);

/* ---- backward (page "M6.1 Routed Capacity", section 0x06F "Single-Device
 * Forward And Backward Integration Contract") ------------------------------
 * Gradients of a scalar loss L with upstream gradient dy = dL/dy, for the
 * forward relation the forward call froze: the chosen ids are metadata (no
 * gradient; the selection bias only chooses), the gates w = rsf s_k / sum_j s_j
 * (or rsf s_k) carry the router's gradient to the chosen experts' logits
 * (dL/dz_k = dL/ds_k s_k (1 - s_k), zero for every other expert), the
 * combine's backward is dU = w dy_r and dL/dw = <dy_r, U>, the gather's
 * adjoint a scatter-add in ascending expert order, and the router, expert,
 * shared and (block) residual paths add at the input.  BF16 layers only
 * (MOE_ERR_UNSUPPORTED otherwise); BF16 operands, FP32 accumulation; the
 * ReLU^2 derivative 2 relu(a) is taken as 2 sqrt(h) from the forward's stored
 * h.  Weight gradients are ADDED to the given FP32 buffers (zero them once
 * per step; a NULL buffer skips that gradient); experts without routes are
 * left untouched (their gradient is zero).                                  */
typedef struct moe_grads {
  float* d_router;    /* [E, d]      */
  float* d_lat_down;  /* [L, d]      latent shapes */
  float* d_lat_up;    /* [d, L]      latent shapes */
  float* d_up;        /* [E, I, de]  */
  float* d_down;      /* [E, de, I]  */
  float* d_sh_up;     /* [S, d]      shared expert */
  float* d_sh_down;   /* [d, S]      shared expert */
  float* d_norm_w;    /* [d]         moe_block_backward only */
} moe_grads_t;

/* Bytes of the backward scratch `bws` for T tokens (0 on an invalid config). */
size_t moe_backward_workspace_bytes(const moe_config_t* cfg, int32_t T);

/* Where the backward scratch keeps its BF16 operands and the gate gradient
 * after a backward call (host arithmetic only), so a caller can inspect them:
 *   MOE_BWS_DU         [T*K, de] bf16  dU = bf16(w dy_r), packed row order
 *   MOE_BWS_DA         [T*K, I]  bf16  da = bf16((dU W_down) * 2 sqrt(h))
 *   MOE_BWS_DZ         [T, K]    FP32  dL/dz of the chosen experts' logits
 *   MOE_BWS_DX_LATENT  [T, L]    bf16  the latent input gradient (latent shapes)
 *   MOE_BWS_DA_SHARED  [T, S]    bf16  the shared expert's da
 *   MOE_BWS_DY_LATENT  [T, L]    bf16  dy_r = bf16(dy W_lu) (latent shapes)  */
enum {
  MOE_BWS_DU = 0, MOE_BWS_DA = 1, MOE_BWS_DZ = 2, MOE_BWS_DX_LATENT = 3, MOE_BWS_DA_SHARED = 4,
  MOE_BWS_DY_LATENT = 5
};
moe_status_t moe_backward_workspace_region(const moe_config_t* cfg, int32_t T, int32_t region,
                                           size_t* offset, size_t* bytes);

/* Backward of moe_layer_forward.  `ws` must be the workspace of a
 * moe_layer_forward call on the same x, weights and T, with no other call on
 * it since (its route tables, h, u, latent rows and shared h are the saved
 * forward state).  topk_ids / topk_w / scores: the forward's router outputs
 * ([T, K] int32, [T, K] FP32, [T, E] FP32; its *_out buffers, or the
 * workspace regions MOE_WS_TOPK_IDS / _TOPK_W / _SCORES when they were NULL).
 *   x [T, d] the forward's input; dy [T, d] act_dtype upstream gradient;
 *   dx [T, d] FP32 out: dL/dx through the router, the experts (and latent
 *   pair) and the shared expert.                                           */
moe_status_t moe_layer_backward(const moe_config_t* cfg, int32_t T, const void* x,
                                const moe_weights_t* w, const void* dy,
                                const int32_t* topk_ids, const float* topk_w, const float* scores,
                                float* dx, const moe_grads_t* grads,
                                const void* ws, size_t ws_bytes, void* bws, size_t bws_bytes,
                                void* stream);

/* Backward of moe_block_forward (out = x + layer(RMSNorm(x))): dout [T, d]
 * act_dtype; dx [T, d] FP32 = dout (the residual) + the RMSNorm's backward of
 * the layer's input gradient; grads->d_norm_w gets dL/dgamma added.  x_norm:
 * the forward's x_norm_out buffer, or NULL when the forward kept the rows in
 * the workspace.  Same state rules as moe_layer_backward.                   */
moe_status_t moe_block_backward(const moe_config_t* cfg, int32_t T, const void* x,
                                const float* norm_w, float norm_eps, const void* x_norm,
                                const moe_weights_t* w, const void* dout,
                                const int32_t* topk_ids, const float* topk_w, const float* scores,
                                float* dx, const moe_grads_t* grads,
                                const void* ws, size_t ws_bytes, void* bws, size_t bws_bytes,
                                void* stream);

/* Synchronises `stream`, copies the device error word of `ws` to *code (host
 * pointer) and returns MOE_ERR_DEVICE if any bit is set, else MOE_OK.         */
moe_status_t moe_get_device_error(const void* ws, void* stream, int32_t* code);

/* Enqueues a clear of the device error word. */
moe_status_t moe_clear_device_error(void* ws, void* stream);

/* How the activations of NVFP4 experts enter their products (process-wide;
 * applies to the calls made after it):
 *   n = -1    the default: three terms on the FP4 tensor path for 8 to 64
 *             tokens, the FP16 path otherwise (the faster one at each size
 *             as measured on GB300)
 *   n = 1..4  the FP4 tensor path: every expert input row and every row of h
 *             is split into n NVFP4 terms, each encoding what the earlier ones
 *             left (E2M1 values, one E4M3 scale per 16 values, one FP32 scale
 *             per row), and the block-scaled FP4 MMA multiplies them with the
 *             NVFP4 weights; n = 1 is plain W4A4.  Each term leaves at most
 *             ~0.18 of the previous residual of a 16-value block, so the
 *             default's n = 3 represents every activation to within ~0.006 of
 *             its block's largest magnitude.  h is stored as BF16.
 *   n = 0     the FP16 path: the weights are decoded to FP16 inside the kernels
 *             and multiplied with FP16 copies of the BF16 activations (exact
 *             for magnitudes up to 65504; a larger activation overflows).
 * Returns the previous setting, or -2 (nothing changed) for n outside -1..4.
 * The block format is the one of page "Nemotron-3.5-Super 120B on an 8 GB
 * GPU", section "The engine, step by step", item 4.                        */
int32_t moe_set_nvfp4_act_terms(int32_t n);

/* The activation terms a call with T tokens uses under the current setting
 * (0: the FP16 path).  Never fails. */
int32_t moe_nvfp4_act_terms_for(int32_t T);

/* Where a workspace for T tokens keeps the layer's route tables, so a caller
 * can read what moe_layer_forward decided (host arithmetic only; no CUDA call).
 * After moe_layer_forward (same cfg, T and workspace) the regions hold:
 *   MOE_WS_COUNTS          [E]     int32  routes per expert
 *   MOE_WS_OFFSETS         [E+1]   int32  exclusive prefix sum of the counts
 *   MOE_WS_ROUTE_TOKEN     [T*K]   int32  token of each packed row
 *   MOE_WS_ROUTE_SLOT      [T*K]   int32  slot of each packed row
 *   MOE_WS_TOKEN_SLOT_ROW  [T, K]  int32  packed row of route (t, k)
 *   MOE_WS_TOPK_IDS        [T, K]  int32  chosen experts   } only when the
 *   MOE_WS_TOPK_W          [T, K]  FP32   routing weights  } matching optional
 *   MOE_WS_LOGITS          [T, E]  FP32   router logits    } output of
 *   MOE_WS_SCORES          [T, E]  FP32   sigmoid scores   } moe_layer_forward is NULL
 *   MOE_WS_X_LATENT        [T, L]  act    latent rows (latent shapes)
 *   MOE_WS_X_PACKED        [T*K, de]      rows packed for the tensor-core path
 *                                         (above 64 BF16 tokens: act_dtype, or
 *                                         FP16 copies of the BF16 values with
 *                                         NVFP4 experts on the FP16 path)
 *   MOE_WS_H               [T*K, I]  act  the experts' ReLU^2 rows h, packed order
 * NVFP4 experts on the FP4 tensor path (moe_set_nvfp4_act_terms n > 0), term
 * j of packed row r of the expert input rows (X) and of h (H):
 *   MOE_WS_X_TERMS / MOE_WS_H_TERMS        [4][T*K][de/2 | I/2] u8  E2M1 codes, even
 *                                           element in the low nibble (terms >= n unused)
 *   MOE_WS_X_TERM_SCALES / _H_TERM_SCALES  [4][T*K][ld] u8  E4M3 scale per 16 values,
 *                                           ld = (K/16 rounded up to 16) for K = de | I
 *   MOE_WS_X_ROW_SCALES / _H_ROW_SCALES    [T*K] FP32  the rows' scale g
 * After moe_block_forward without x_norm_out:
 *   MOE_WS_X_NORM          [T, d]  act    the RMSNorm rows xn
 * *offset receives the region's byte offset from the workspace start, *bytes
 * its size.  MOE_ERR_INVALID_ARG for an unknown region or T < 0.           */
enum {
  MOE_WS_COUNTS = 0, MOE_WS_OFFSETS = 1, MOE_WS_ROUTE_TOKEN = 2, MOE_WS_ROUTE_SLOT = 3,
  MOE_WS_TOKEN_SLOT_ROW = 4, MOE_WS_TOPK_IDS = 5, MOE_WS_TOPK_W = 6, MOE_WS_LOGITS = 7,
  MOE_WS_SCORES = 8, MOE_WS_X_LATENT = 9, MOE_WS_X_PACKED = 10, MOE_WS_H = 11, MOE_WS_X_TERMS = 12,
  MOE_WS_X_TERM_SCALES = 13, MOE_WS_X_ROW_SCALES = 14, MOE_WS_H_TERMS = 15, MOE_WS_H_TERM_SCALES = 16,
  MOE_WS_H_ROW_SCALES = 17, MOE_WS_X_NORM = 18
};
moe_status_t moe_workspace_region(const moe_config_t* cfg, int32_t T, int32_t region, size_t* offset,
                                  size_t* bytes);

/* Number of kernel launches this library has enqueued in this process (a host
 * counter, incremented once per kernel launch; memset and copy operations are
 * not counted).  Never fails. */
int64_t moe_launch_count(void);

/* Router step that allocates nothing and takes no workspace.  The pages have
 * no counterpart: this serves callers that cannot allocate device memory at
 * call time, such as code running after a host framework's memory pool has
 * claimed the device, serving loops that forbid allocation once started, or
 * work enqueued where cudaMalloc is not permitted.  Same arguments and
 * results as moe_router without logits/scores outputs (the same kernels,
 * bit-identical results); its scratch (logits, scores, the BF16 split of the
 * router matrix and the four K-split logit slabs used above 64 BF16 tokens,
 * and the error word) lives in a static device array of
 * MOE_NOALLOC_MAX_ROUTER_ELEMS * 24 + MOE_NOALLOC_MAX_SPLIT_ELEMS * 2 + 256
 * bytes (about 17 MiB) that every GPU loading this library keeps until exit.
 *   - Returns MOE_ERR_WORKSPACE, before enqueuing anything, when
 *     T * n_experts > MOE_NOALLOC_MAX_ROUTER_ELEMS, or when T > 64 BF16
 *     tokens need the split router matrix and 3 * n_experts * d_model >
 *     MOE_NOALLOC_MAX_SPLIT_ELEMS.
 *   - The first call on a device looks the array up (cudaGetSymbolAddress,
 *     once per device, with that device current) and keeps the address for
 *     the life of the process: it assumes the device's primary context is
 *     never reset (cudaDeviceReset) while the library is loaded.
 *   - All calls share the array: calls whose work overlaps on the GPU race.
 *     Each call clears the error word first; device error bits are not
 *     reported by this entry point.
 *   - Calls no allocation routine (no cudaMalloc/cudaFree).                  */
#define MOE_NOALLOC_MAX_ROUTER_ELEMS 131072
#define MOE_NOALLOC_MAX_SPLIT_ELEMS 7340032
moe_status_t moe_router_noalloc(const moe_config_t* cfg, int32_t T, const void* x,
                                const float* w_router, const float* router_bias,
                                int32_t* topk_ids, float* topk_w, void* stream);

/* End-to-end convenience call with HOST buffers: copies x_host [T, d] to
 * x_dev, runs moe_layer_forward, copies y to y_host and synchronises the
 * stream.  x_dev / y_dev / ws are caller-owned device buffers; the host
 * buffers should be pinned for asynchronous copies.                          */
moe_status_t moe_layer_forward_host(const moe_config_t* cfg, int32_t T, const void* x_host,
                                    void* x_dev, const moe_weights_t* w, void* y_dev,
                                    void* y_host, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
