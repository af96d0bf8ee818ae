// moe_router_noalloc: the router step for callers that cannot allocate device
// memory, e.g. code that runs after its host framework's pool has claimed all
// device memory, runtimes that forbid allocation once serving starts, or code
// enqueued where cudaMalloc is not permitted.  The scratch the router needs
// between its kernels (logits, scores, the K-split partial logits, the split
// router matrix, the device error word) lives in a fixed static device array of
// this file instead of a caller workspace.
//
// Properties the caller must know:
//  - The array (MOE_NOALLOC_MAX_ROUTER_ELEMS * 24 + MOE_NOALLOC_MAX_SPLIT_ELEMS
//    * 2 + 256 bytes, about 17 MiB) exists on every GPU that loads the
//    library, for the life of the process.
//  - It computes exactly what moe_router computes, by the same kernels: for
//    more than 64 BF16 tokens that includes the BF16 split of the router
//    matrix (E * 3d BF16 values) and the logits split over up to four K parts
//    (four logit-sized slabs), both held in the array.
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, with that device current).  The
//    address is kept for the life of the process: it assumes the device's primary context is never
//    reset (after cudaDeviceReset the array would have to be looked up again).
//  - Every call shares the one array: two calls whose work overlaps on the GPU
//    (different streams, no ordering between them) race on it.  The error
//    word is cleared at the start of every call; logits and scores are fully
//    rewritten by each call before they are read, and so is the split router
//    matrix when it is used.
//  - The error word stays in the array: this entry point does not report
//    device-side error bits.
#include "internal.h"

#include <mutex>

namespace {

constexpr int64_t kMaxElems = MOE_NOALLOC_MAX_ROUTER_ELEMS;
constexpr int64_t kMaxSplit = MOE_NOALLOC_MAX_SPLIT_ELEMS;
constexpr size_t kHeaderBytes = 256;

// [0, 256): error word;  logits [kMaxElems] f32;  scores [kMaxElems] f32;
// K-split logit slabs [kRouterParts * kMaxElems] f32;  split router matrix
// [kMaxSplit] bf16
static __device__ __align__(256) unsigned char
    g_router_scratch[kHeaderBytes + (2 + moe::kRouterParts) * kMaxElems * sizeof(float) + kMaxSplit * 2];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static array on the current device (looked up once per device).
moe_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_router_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_router_noalloc(const moe_config_t* cfg, int32_t T, const void* x,
                                           const float* w_router, const float* router_bias, int32_t* topk_ids,
                                           float* topk_w, void* stream) {
  moe_status_t st = moe_check_config(cfg);
  if (st != MOE_OK) return st;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if ((int64_t)T * cfg->n_experts > kMaxElems) return MOE_ERR_WORKSPACE;   // beyond the static scratch
  // the same condition as the router's tensor-core path (d_model % 64 == 0
  // holds for every valid configuration)
  const bool needs_split = cfg->act_dtype == MOE_DT_BF16 && T > 64 && cfg->n_experts % 32 == 0;
  if (needs_split && (int64_t)3 * cfg->n_experts * cfg->d_model > kMaxSplit) return MOE_ERR_WORKSPACE;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_ids) || !aligned16(topk_w) ||
      (router_bias && !aligned16(router_bias)))
    return MOE_ERR_INVALID_ARG;
  void* base = nullptr;
  if ((st = scratch_address(&base)) != MOE_OK) return st;
  int32_t* err = reinterpret_cast<int32_t*>(base);
  float* logits = reinterpret_cast<float*>(reinterpret_cast<char*>(base) + kHeaderBytes);
  float* scores = logits + kMaxElems;
  float* parts = scores + kMaxElems;
  void* split = reinterpret_cast<void*>(parts + moe::kRouterParts * kMaxElems);
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  int nparts = 1;
  if (moe::launch_router_logits(x, cfg->act_dtype, T, cfg->d_model, w_router, cfg->n_experts, logits, s, split,
                                T > 64 ? parts : nullptr, &nparts) != cudaSuccess)
    return MOE_ERR_CUDA;
  const bool ks = nparts > 1;
  if (moe::launch_router_select(ks ? parts : logits, nparts, (int64_t)T * cfg->n_experts, ks ? logits : nullptr, T,
                                cfg->n_experts, router_bias, cfg->n_group, cfg->topk_group, cfg->top_k,
                                cfg->norm_topk_prob, cfg->routed_scaling_factor, scores, topk_ids, topk_w, err,
                                s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
