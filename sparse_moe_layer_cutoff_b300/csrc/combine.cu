// latent_norm + weighted fusion: c[t] = gamma * sum_k w[t,k] * y_tk / sqrt(mean(y_tk^2) + eps),
// y_tk = y[inv[t, k]] ("KimiK3的StableLatentMoE架构解析", ¶"具体前向流程" and ¶"第二":
// RMSNorm on each expert's latent output, before the weighted fusion and up_proj).
// The other placement ("Vue d'ensemble de l'architecture", "Par où l'information passe",
// step f: "RMSNorm + W_up" as one step) normalises the weighted sum once:
//   c[t] = gamma * s / sqrt(mean(s^2) + eps),  s = sum_k w[t,k] * y_tk.
//
// HBM-bound: each token reads its K latent rows once from DRAM (the second pass over them
// hits L1/L2) and writes one latent row.  One block per token; phase 1 gives every k its
// scale w / rms with one warp per row; phase 2 sums the K rows in fixed k order with
// 16-byte vector loads.  With the norm on the sum, phase 1 is just w, phase 2 parks the fp32
// sum in shared memory while the block reduces its sum of squares, and phase 3 scales it.
// Block size (combine_threads): at K = 16, latent 3584 the per-expert norm runs 512 threads,
// all 16 rows in phase 1 at once; its output does not depend on the block size.
#include "common.cuh"
#include "internal.h"

namespace lmoe {

constexpr int kCombThreads = 512;   // largest block

// Threads per block.  Per-expert norm: one warp per expert row (phase 1) or one 16-byte chunk
// per thread (phase 2), whichever is more, up to 512.  Norm on the sum (no phase 1): up to 256,
// two chunks per thread at latent 3584 (measured faster there than 448 threads with one).
int combine_threads(int top_k, int latent, int vec, bool norm_sum) {
  int n = !norm_sum && top_k * 32 > latent / vec ? top_k * 32 : latent / vec;
  n = (n + 31) / 32 * 32;
  const int cap = norm_sum ? 256 : kCombThreads;
  return n < 64 ? 64 : n > cap ? cap : n;
}

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

template <typename T, bool NORM_SUM>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const CombineArgs a) {
  constexpr int V = Vec<T>::n;
  __shared__ float s_scale[kMaxTopK];
  __shared__ long long s_row[kMaxTopK];
  __shared__ float s_part[kCombThreads / 32];
  extern __shared__ float s_sum[];   // [latent] fp32 weighted sum (NORM_SUM only)
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const T* y = static_cast<const T*>(a.y);
  const int L = a.latent;

  for (int k = threadIdx.x; k < a.top_k; k += blockDim.x) {
    s_row[k] = (long long)a.inv[(long long)t * a.top_k + k] * L;
    if constexpr (NORM_SUM) s_scale[k] = a.w[(long long)t * a.top_k + k];
  }
  __syncthreads();
  if constexpr (!NORM_SUM) {
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
  }
  const T* gamma = static_cast<const T*>(a.gamma);
  T* out = static_cast<T*>(a.cat) + (long long)t * a.ldc;
  float ss = 0.f;
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
    if constexpr (NORM_SUM) {
#pragma unroll
      for (int q = 0; q < V; ++q) {
        s_sum[i + q] = acc[q];
        ss = fmaf(acc[q], acc[q], ss);
      }
    } else {
      float gv[V];
      load_vec(gamma + i, gv);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] *= gv[q];
      store_vec(out + i, acc);
    }
  }
  if constexpr (NORM_SUM) {
    ss = warp_sum(ss);
    if (lane == 0) s_part[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nw; ++w) tot += s_part[w];   // fixed order: same value in every thread
    const float inv_rms = 1.0f / sqrtf(tot / (float)L + a.eps);
    // every thread reads back only the elements it wrote above
    for (int i = threadIdx.x * V; i < L; i += blockDim.x * V) {
      float acc[V], gv[V];
      load_vec(gamma + i, gv);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = s_sum[i + q] * inv_rms * gv[q];
      store_vec(out + i, acc);
    }
  }
}

size_t combine_smem_bytes(int latent, bool norm_sum) { return norm_sum ? (size_t)latent * sizeof(float) : 0; }

cudaError_t prepare_combine(int latent, bool norm_sum) {
  const size_t smem = combine_smem_bytes(latent, norm_sum);
  if (smem <= 48 * 1024) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(combine_kernel<bf16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(combine_kernel<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e;
}

cudaError_t launch_combine(const CombineArgs& a, bool bf16_, cudaStream_t st) {
  if (a.bt <= 0) return cudaSuccess;
  const size_t smem = combine_smem_bytes(a.latent, a.norm_sum);
  const int nt = combine_threads(a.top_k, a.latent, bf16_ ? Vec<bf16>::n : Vec<float>::n, a.norm_sum);
  if (a.norm_sum) {
    if (bf16_) combine_kernel<bf16, true><<<a.bt, nt, smem, st>>>(a);
    else combine_kernel<float, true><<<a.bt, nt, smem, st>>>(a);
  } else {
    if (bf16_) combine_kernel<bf16, false><<<a.bt, nt, 0, st>>>(a);
    else combine_kernel<float, false><<<a.bt, nt, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace lmoe
