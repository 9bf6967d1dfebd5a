// Validation of the routing index buffers (check mode and lmoe_debug_check_segments).
//
// The expert segments are a stable counting sort of the bt*K (token, k) pairs by expert
// ("KimiK3的StableLatentMoE架构解析", ¶"具体前向流程": tokens are grouped by expert for the
// GroupedExperts).  Every later kernel indexes memory through them, so a check mode verifies
// them on the device before any of those kernels runs:
//   * every id idx[t, k] is in [0, E) and the K ids of a token are distinct;
//   * offsets[0] = 0, offsets[E] = bt*K, counts[e] = offsets[e+1] - offsets[e] >= 0;
//   * the slot s = inv[t, k] lies in expert idx[t, k]'s segment and perm[s] = t.
// Distinct ids put a token's K slots in K different segments, and perm[s] names one token per
// slot, so inv is injective on the bt*K pairs and, with bt*K slots, a bijection.
// A failed check sets kStatusAssert in the status word (no trap); every index is bounds-checked
// before it is used as an address.
#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

__global__ void __launch_bounds__(256)
validate_segments_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ counts,
                         const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm,
                         const int32_t* __restrict__ inv, int bt, int top_k, int n_experts,
                         uint32_t* __restrict__ status) {
  const long long pairs = (long long)bt * top_k;
  bool bad = false;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (tid == 0) bad |= offsets[0] != 0 || (long long)offsets[n_experts] != pairs;
  for (long long e = tid; e < n_experts; e += stride) {
    const int n = offsets[e + 1] - offsets[e];
    bad |= n < 0 || counts[e] != n;
  }
  for (long long p = tid; p < pairs; p += stride) {
    const int t = (int)(p / top_k);
    const int k = (int)(p - (long long)t * top_k);
    const int e = idx[p];
    if (e < 0 || e >= n_experts) {
      bad = true;
      continue;
    }
    for (int j = 0; j < k; ++j) bad |= idx[(long long)t * top_k + j] == e;
    const int s = inv[p];
    if (s < offsets[e] || s >= offsets[e + 1] || s < 0 || (long long)s >= pairs) {
      bad = true;
      continue;
    }
    bad |= perm[s] != t;
  }
  if (bad) atomicOr(status, kStatusAssert);
}

}  // namespace

cudaError_t launch_validate_segments(const int32_t* idx, const int32_t* counts, const int32_t* offsets,
                                     const int32_t* perm, const int32_t* inv, int bt, int top_k, int n_experts,
                                     uint32_t* status, int sm_count, cudaStream_t st) {
  if (bt <= 0) return cudaSuccess;
  const long long pairs = (long long)bt * top_k;
  const long long work = pairs > n_experts ? pairs : n_experts;
  long long blocks = (work + 255) / 256;
  if (blocks > 8LL * sm_count) blocks = 8LL * sm_count;
  validate_segments_kernel<<<(int)blocks, 256, 0, st>>>(idx, counts, offsets, perm, inv, bt, top_k, n_experts,
                                                        status);
  return cudaGetLastError();
}

}  // namespace lmoe
