// latent_norm + weighted fusion: c[t] = gamma * sum_k w[t,k] * y_tk / sqrt(mean(y_tk^2) + eps),
// y_tk = y[inv[t, k]] ("KimiK3的StableLatentMoE架构解析", ¶"具体前向流程" and ¶"第二":
// RMSNorm on each expert's latent output, before the weighted fusion and up_proj).
//
// HBM-bound: each token reads its K latent rows once from DRAM (the second pass over them
// hits L1/L2) and writes one latent row.  One block per token; phase 1 gives every k its
// scale w / rms with one warp per row; phase 2 sums the K rows in fixed k order with
// 16-byte vector loads.
#include "common.cuh"
#include "internal.h"

namespace lmoe {

constexpr int kCombThreads = 256;

template <typename T> struct Vec;
template <> struct Vec<bf16> { static constexpr int n = 8; };
template <> struct Vec<float> { static constexpr int n = 4; };

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float* v) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 2) {
    const bf16* h = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __bfloat162float(h[i]);
  } else {
    const float* f = reinterpret_cast<const float*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = f[i];
  }
}

template <typename T>
__device__ __forceinline__ void store_vec(T* p, const float* v) {
  uint4 raw;
  if constexpr (sizeof(T) == 2) {
    bf16* h = reinterpret_cast<bf16*>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = __float2bfloat16_rn(v[i]);
  } else {
    float* f = reinterpret_cast<float*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = v[i];
  }
  *reinterpret_cast<uint4*>(p) = raw;
}

template <typename T>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const CombineArgs a) {
  constexpr int V = Vec<T>::n;
  __shared__ float s_scale[kMaxTopK];
  __shared__ long long s_row[kMaxTopK];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const T* y = static_cast<const T*>(a.y);
  const int L = a.latent;

  for (int k = threadIdx.x; k < a.top_k; k += blockDim.x)
    s_row[k] = (long long)a.inv[(long long)t * a.top_k + k] * L;
  __syncthreads();
  for (int k = warp; k < a.top_k; k += nw) {
    const T* row = y + s_row[k];
    float ss = 0.f;
    for (int i = lane * V; i < L; i += 32 * V) {
      float v[V];
      load_vec(row + i, v);
#pragma unroll
      for (int q = 0; q < V; ++q) ss = fmaf(v[q], v[q], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) s_scale[k] = a.w[(long long)t * a.top_k + k] / sqrtf(ss / (float)L + a.eps);
  }
  __syncthreads();
  const T* gamma = static_cast<const T*>(a.gamma);
  T* out = static_cast<T*>(a.cat) + (long long)t * a.ldc;
  for (int i = threadIdx.x * V; i < L; i += blockDim.x * V) {
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
    for (int k = 0; k < a.top_k; ++k) {
      float v[V];
      load_vec(y + s_row[k] + i, v);
      const float sc = s_scale[k];
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = fmaf(sc, v[q], acc[q]);
    }
    float gv[V];
    load_vec(gamma + i, gv);
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] *= gv[q];
    store_vec(out + i, acc);
  }
}

cudaError_t launch_combine(const CombineArgs& a, bool bf16_, cudaStream_t st) {
  if (a.bt <= 0) return cudaSuccess;
  if (bf16_) combine_kernel<bf16><<<a.bt, kCombThreads, 0, st>>>(a);
  else combine_kernel<float><<<a.bt, kCombThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace lmoe
