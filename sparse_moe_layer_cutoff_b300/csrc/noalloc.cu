// Expert segmentation without any allocation by the library.
//
// Some callers cannot let a library call cudaMalloc: their device memory is owned by
// another allocator (for example a framework's caching pool that has already reserved
// the free HBM, where a stray cudaMalloc fails or fragments it), or they run on a
// latency-critical path where cudaMalloc's implicit device synchronisation is not
// acceptable.  lmoe_segments_noalloc serves them: the caller passes its inputs and
// outputs, and the only working memory, the per-block expert counts of the counting
// sort, lives in the fixed device array below, which every GPU that loads this library
// holds until the process exits.
#include <cuda.h>

#include <mutex>

#include "../../include/lmoe.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = 4u << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t lmoe_noalloc_scratch[kScratchBytes / sizeof(int32_t)];

// Per device: the array's device address and the context it was looked up in (a device reset
// creates a new primary context, whose address and kernel attributes must be set up again).
struct ScratchEntry {
  CUcontext ctx;
  int32_t* ptr;
};

std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices];   // the host-side name of the array is not its device address

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    cudaGetLastError();
  }
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// With the device current: the array's device address, looked up once per device and
// context (the lookup also makes the runtime create the device's context if needed).
lmoe_status scratch_for_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchEntry& ent = g_scratch[dev];
  const CUcontext cur = current_context();
  if (!ent.ptr || !cur || ent.ctx != cur) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, lmoe_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return LMOE_ERR_CUDA;
    }
    if (lmoe::route_tail_prepare() != cudaSuccess) {
      cudaGetLastError();
      return LMOE_ERR_CUDA;
    }
    ent.ptr = static_cast<int32_t*>(p);
    ent.ctx = current_context();
  }
  *out = ent.ptr;
  return LMOE_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" lmoe_status lmoe_segments_noalloc(const int32_t* topk_idx, int32_t bt, int32_t top_k,
                                             int32_t n_experts, int32_t* expert_counts, int32_t* offsets,
                                             int32_t* perm, int32_t* inv, lmoe_stream stream) {
  if (bt < 0 || top_k < 1 || n_experts < top_k) return LMOE_ERR_INVALID_ARG;
  if (n_experts > lmoe::kMaxExperts || top_k > lmoe::kMaxTopK) return LMOE_ERR_UNSUPPORTED;
  if ((long long)bt * top_k >= (1LL << 31)) return LMOE_ERR_UNSUPPORTED;
  // scratch layout: per-block counts [nblk][E], counts [E], tile prefix [E + 1]
  const long long nblk = ((long long)bt + lmoe::kSegTokens - 1) / lmoe::kSegTokens;
  const long long need = (nblk * n_experts + 2LL * n_experts + 1) * (long long)sizeof(int32_t);
  if (need > (long long)kScratchBytes) return LMOE_ERR_UNSUPPORTED;
  if (bt == 0) return LMOE_OK;
  const void* ptrs[] = {topk_idx, expert_counts, offsets, perm, inv};
  for (const void* p : ptrs)
    if (!p || !aligned4(p)) return LMOE_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  lmoe_status s = scratch_for_current_device(&scratch);
  if (s != LMOE_OK) return s;
  // Every block-count entry the chain reads is written earlier in the same call, so no
  // part of the scratch has to start at zero.
  int32_t* block_cnt = scratch;
  int32_t* counts = scratch + nblk * n_experts;
  int32_t* mtile_off = counts + n_experts;
  cudaError_t e = lmoe::launch_segments(topk_idx, bt, top_k, n_experts, block_cnt, counts, offsets, mtile_off,
                                        perm, inv, expert_counts, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}
