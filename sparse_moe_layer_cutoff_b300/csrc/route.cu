// Router kernels after the logits GEMM: Quantile Balancing cutoffs, top-K with combine
// weights, and the stable per-expert segmentation of the (token, k) pairs.
//
// "KimiK3的StableLatentMoE架构解析" (tech.news18a.com), ¶"第三": a per-expert cutoff alpha
// steers each expert's token count toward its quantile target, with sigmoid gating;
// ¶"具体前向流程": top-16 experts per token, then GroupedExperts.  The cutoff is the
// (1 - K/E) linear-interpolation quantile of the expert's sigmoid scores over the batch;
// selection is the top-K of (score - cutoff), ties to the lower expert index; combine
// weights are the chosen raw scores renormalised.
#include "common.cuh"
#include "internal.h"

namespace lmoe {

// ------------------------------------------------------------------------------------
// alpha_e: radix-select the order statistics j and j+1 of the logits column e (sigmoid is
// monotone, so the sorted scores are the sigmoid of the sorted logits), then interpolate
// in score space in fp64.  One block per expert; the column is contiguous in logits^T.
// ------------------------------------------------------------------------------------
constexpr int kCutoffThreads = 256;

__global__ void __launch_bounds__(kCutoffThreads)
qb_cutoff_kernel(const float* __restrict__ logits_t, int bt, int n_experts, int top_k,
                 double* __restrict__ alpha) {
  const int e = blockIdx.x;
  const float* col = logits_t + (size_t)e * bt;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_bucket, s_below;
  __shared__ uint32_t s_cnt_le, s_min_gt;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const long long num = (long long)(bt - 1) * (long long)(n_experts - top_k);
  const long long j = num / n_experts;
  const double frac = (double)(num - j * n_experts) / (double)n_experts;

  uint32_t prefix = 0, mask = 0;
  uint32_t rank = (uint32_t)j;  // rank of the target among the keys matching prefix
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < bt; i += blockDim.x) {
      uint32_t k = f32_to_key(col[i]);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t local[8], sum = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) { local[b] = hist[lane * 8 + b]; sum += local[b]; }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      uint32_t excl = incl - sum;
      if (rank >= excl && rank < incl) {
        uint32_t c = excl;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (rank < c + local[b]) { s_bucket = lane * 8 + b; s_below = c; break; }
          c += local[b];
        }
      }
    }
    __syncthreads();
    prefix |= s_bucket << shift;
    mask |= 255u << shift;
    rank -= s_below;
    __syncthreads();
  }
  const uint32_t kj = prefix;

  // v_{j+1}: equal to v_j when at least j+2 keys are <= v_j, else the smallest key above it.
  if (tid == 0) { s_cnt_le = 0; s_min_gt = 0xffffffffu; }
  __syncthreads();
  uint32_t cnt = 0, mn = 0xffffffffu;
  for (int i = tid; i < bt; i += blockDim.x) {
    uint32_t k = f32_to_key(col[i]);
    if (k <= kj) ++cnt; else mn = min(mn, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (lane == 0) { atomicAdd(&s_cnt_le, cnt); atomicMin(&s_min_gt, mn); }
  __syncthreads();
  if (tid == 0) {
    const double vj = sigmoid_f64((double)key_to_f32(kj));
    double a = vj;
    if (j + 1 < bt) {
      const uint32_t kj1 = ((long long)s_cnt_le >= j + 2) ? kj : s_min_gt;
      const double vj1 = sigmoid_f64((double)key_to_f32(kj1));
      // no fused multiply-add: the same rounding as a plain a + f * (b - a)
      a = __dadd_rn(vj, __dmul_rn(frac, __dsub_rn(vj1, vj)));
    }
    alpha[e] = a;
  }
}

// ------------------------------------------------------------------------------------
// Top-K per token: one warp per token.  Keys s - alpha (fp64) live in shared memory; each
// lane keeps the best of its own experts (e = lane + 32 i) and the warp picks the best of
// the lane bests K times.  Order: key descending, then expert index ascending.
// ------------------------------------------------------------------------------------
constexpr int kTopkWarps = 4;

__device__ __forceinline__ bool topk_better(bool v1, double k1, int e1, bool v2, double k2, int e2) {
  if (v1 != v2) return v1;
  if (!v1) return false;
  return k1 > k2 || (k1 == k2 && e1 < e2);
}

__global__ void __launch_bounds__(kTopkWarps * 32)
topk_kernel(const float* __restrict__ logits, const double* __restrict__ alpha, int bt,
            int n_experts, int top_k, int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  extern __shared__ double smem_d[];
  double* s_alpha = smem_d;                                        // [E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  double* keys = smem_d + n_experts + (size_t)warp * n_experts;   // [E] per warp
  double* chosen_s = smem_d + (size_t)(kTopkWarps + 1) * n_experts + warp * 64;  // [K<=64]
  uint8_t* taken = reinterpret_cast<uint8_t*>(smem_d + (size_t)(kTopkWarps + 1) * n_experts +
                                              kTopkWarps * 64) + (size_t)warp * n_experts;

  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) s_alpha[e] = alpha[e];
  __syncthreads();

  for (int t = blockIdx.x * kTopkWarps + warp; t < bt; t += gridDim.x * kTopkWarps) {
    const float* lrow = logits + (size_t)t * n_experts;
    bool bv = false; double bk = 0.0; int be = 0;
    for (int e = lane; e < n_experts; e += 32) {
      double kv = sigmoid_f64((double)lrow[e]) - s_alpha[e];
      keys[e] = kv;
      taken[e] = 0;
      if (!bv || kv > bk) { bv = true; bk = kv; be = e; }
    }
    __syncwarp();
    for (int k = 0; k < top_k; ++k) {
      bool v = bv; double kk = bk; int ee = be;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        bool v2 = __shfl_down_sync(0xffffffffu, v, o);
        double k2 = __shfl_down_sync(0xffffffffu, kk, o);
        int e2 = __shfl_down_sync(0xffffffffu, ee, o);
        if (lane + o < 32 && topk_better(v2, k2, e2, v, kk, ee)) { v = v2; kk = k2; ee = e2; }
      }
      ee = __shfl_sync(0xffffffffu, ee, 0);
      if (lane == 0) idx_out[(size_t)t * top_k + k] = ee;
      if ((ee & 31) == lane) {
        taken[ee] = 1;
        bv = false;
        for (int e = lane; e < n_experts; e += 32) {
          if (taken[e]) continue;
          double kv = keys[e];
          if (!bv || kv > bk) { bv = true; bk = kv; be = e; }
        }
      }
      if (lane == 0) chosen_s[k] = (double)ee;  // expert id, converted back below
      __syncwarp();
    }
    // combine weights: chosen raw scores over their sum (summed in k order, fp64)
    for (int k = lane; k < top_k; k += 32) {
      int e = (int)chosen_s[k];
      chosen_s[k] = sigmoid_f64((double)lrow[e]);
    }
    __syncwarp();
    double total = 0.0;
    for (int k = 0; k < top_k; ++k) total = total + chosen_s[k];
    for (int k = lane; k < top_k; k += 32)
      w_out[(size_t)t * top_k + k] = (float)(chosen_s[k] / total);
    __syncwarp();
  }
}

size_t topk_smem_bytes(int n_experts) {
  return (size_t)(kTopkWarps + 1) * n_experts * sizeof(double) + kTopkWarps * 64 * sizeof(double) +
         (size_t)kTopkWarps * n_experts;
}

// ------------------------------------------------------------------------------------
// Segments.  The bt*K pairs in (t, k) order are split into chunks of kSegTokens tokens,
// one block each; inside a block each warp takes a contiguous run of pairs.  The rank of
// a pair among the earlier pairs with the same expert is built from warp match masks and
// per-warp counters, so the result is a stable counting sort, independent of timing.
// ------------------------------------------------------------------------------------
constexpr int kSegThreads = 256;
constexpr int kSegWarps = kSegThreads / 32;

// Per-warp counts (and, when want_pos, each pair's rank inside its warp) for one chunk.
// cnt: [kSegWarps][E] shared counters, zeroed by the caller.
template <bool kWantPos>
__device__ __forceinline__ void seg_warp_pass(const int32_t* __restrict__ idx, long long p_begin,
                                              long long p_end, int per_warp, int n_experts,
                                              uint32_t* cnt, uint32_t* pos_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* my = cnt + (size_t)warp * n_experts;
  const long long w0 = p_begin + (long long)warp * per_warp;
  const unsigned lt = (1u << lane) - 1u;
  for (int r = 0; r < per_warp; r += 32) {
    long long p = w0 + r + lane;
    bool ok = (r + lane < per_warp) && (p < p_end);
    int e = ok ? idx[p] : -1;
    if (ok && (e < 0 || e >= n_experts)) e = -1;  // out-of-range id: counted nowhere
    unsigned m = __match_any_sync(0xffffffffu, e);
    uint32_t rank = __popc(m & lt);
    uint32_t base = (e >= 0) ? my[e] : 0u;
    __syncwarp();
    if (e >= 0 && (m & lt) == 0) my[e] = base + __popc(m);
    __syncwarp();
    if (kWantPos) pos_out[r >> 5] = (e >= 0) ? base + rank : 0xffffffffu;
  }
}

__global__ void __launch_bounds__(kSegThreads)
seg_count_kernel(const int32_t* __restrict__ idx, int bt, int top_k, int n_experts,
                 int32_t* __restrict__ block_cnt /* [nblk][E] */) {
  extern __shared__ uint32_t cnt[];  // [kSegWarps][E]
  for (int i = threadIdx.x; i < kSegWarps * n_experts; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const long long p_begin = (long long)blockIdx.x * kSegTokens * top_k;
  const long long p_end = min((long long)bt * top_k, p_begin + (long long)kSegTokens * top_k);
  const int per_warp = (kSegTokens * top_k) / kSegWarps;
  seg_warp_pass<false>(idx, p_begin, p_end, per_warp, n_experts, cnt, nullptr);
  __syncthreads();
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
    uint32_t s = 0;
    for (int w = 0; w < kSegWarps; ++w) s += cnt[(size_t)w * n_experts + e];
    block_cnt[(size_t)blockIdx.x * n_experts + e] = (int32_t)s;
  }
}

// One block: per-expert counts, segment offsets, per-block bases and the m-tile prefix
// used by the grouped GEMM schedulers.
__global__ void __launch_bounds__(1024)
seg_scan_kernel(int32_t* __restrict__ block_cnt /* in: counts, out: bases */, int nblk,
                int n_experts, int tile_m, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets /* [E+1] */, int32_t* __restrict__ mtile_off /* [E+1] */,
                int32_t* __restrict__ user_counts) {
  extern __shared__ int32_t sm_i[];
  int32_t* s_cnt = sm_i;                 // [E]
  int32_t* s_mt = sm_i + n_experts;      // [E]
  __shared__ int32_t s_warp[2][32];
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
    int32_t s = 0;
    for (int b = 0; b < nblk; ++b) s += block_cnt[(size_t)b * n_experts + e];
    s_cnt[e] = s;
    s_mt[e] = (s + tile_m - 1) / tile_m;
    counts[e] = s;
    if (user_counts) user_counts[e] = s;
  }
  __syncthreads();
  // exclusive scans of s_cnt and s_mt: each thread owns a contiguous run of experts
  const int per = (n_experts + blockDim.x - 1) / blockDim.x;
  const int e0 = min(n_experts, (int)threadIdx.x * per), e1 = min(n_experts, e0 + per);
  int32_t a = 0, b = 0;
  for (int e = e0; e < e1; ++e) { a += s_cnt[e]; b += s_mt[e]; }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += va; ib += vb; }
  }
  if (lane == 31) { s_warp[0][warp] = ia; s_warp[1][warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x / 32;
    int32_t wa = lane < nw ? s_warp[0][lane] : 0, wb = lane < nw ? s_warp[1][lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t va = __shfl_up_sync(0xffffffffu, wa, o), vb = __shfl_up_sync(0xffffffffu, wb, o);
      if (lane >= o) { wa += va; wb += vb; }
    }
    if (lane < nw) { s_warp[0][lane] = wa; s_warp[1][lane] = wb; }
  }
  __syncthreads();
  int32_t ra = ia - a + (warp > 0 ? s_warp[0][warp - 1] : 0);
  int32_t rb = ib - b + (warp > 0 ? s_warp[1][warp - 1] : 0);
  for (int e = e0; e < e1; ++e) {
    offsets[e] = ra; mtile_off[e] = rb;
    // per-block bases inside the segment
    int32_t run = ra;
    for (int blk = 0; blk < nblk; ++blk) {
      int32_t c = block_cnt[(size_t)blk * n_experts + e];
      block_cnt[(size_t)blk * n_experts + e] = run;
      run += c;
    }
    ra += s_cnt[e]; rb += s_mt[e];
  }
  if (threadIdx.x == blockDim.x - 1) {
    // the last thread's running values are the totals
    offsets[n_experts] = ra;
    mtile_off[n_experts] = rb;
  }
}

__global__ void __launch_bounds__(kSegThreads)
seg_scatter_kernel(const int32_t* __restrict__ idx, int bt, int top_k, int n_experts,
                   const int32_t* __restrict__ block_base /* [nblk][E] */,
                   int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  extern __shared__ uint32_t cnt[];  // [kSegWarps][E]
  for (int i = threadIdx.x; i < kSegWarps * n_experts; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const long long p_begin = (long long)blockIdx.x * kSegTokens * top_k;
  const long long p_end = min((long long)bt * top_k, p_begin + (long long)kSegTokens * top_k);
  const int per_warp = (kSegTokens * top_k) / kSegWarps;
  uint32_t pos[kSegTokens * 64 / kSegWarps / 32];  // per_warp / 32 rounds at most
  seg_warp_pass<true>(idx, p_begin, p_end, per_warp, n_experts, cnt, pos);
  __syncthreads();
  // exclusive prefix over warps, per expert
  for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
    uint32_t run = 0;
    for (int w = 0; w < kSegWarps; ++w) {
      uint32_t c = cnt[(size_t)w * n_experts + e];
      cnt[(size_t)w * n_experts + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long w0 = p_begin + (long long)warp * per_warp;
  for (int r = 0; r < per_warp; r += 32) {
    long long p = w0 + r + lane;
    if (r + lane >= per_warp || p >= p_end) continue;
    int e = idx[p];
    if (e < 0 || e >= n_experts) continue;
    int32_t slot = block_base[(size_t)blockIdx.x * n_experts + e] +
                   (int32_t)cnt[(size_t)warp * n_experts + e] + (int32_t)pos[r >> 5];
    perm[slot] = (int32_t)(p / top_k);
    inv[p] = slot;
  }
}

// ------------------------------------------------------------------------------------
// Host launchers.
// ------------------------------------------------------------------------------------
cudaError_t launch_route_tail(const RouteArgs& a, cudaStream_t st) {
  if (a.bt <= 0) return cudaSuccess;
  qb_cutoff_kernel<<<a.n_experts, kCutoffThreads, 0, st>>>(a.logits_t, a.bt, a.n_experts, a.top_k,
                                                          a.alpha);
  const size_t tk_smem = topk_smem_bytes(a.n_experts);
  int tk_grid = (a.bt + kTopkWarps - 1) / kTopkWarps;
  if (tk_grid > 148 * 16) tk_grid = 148 * 16;
  topk_kernel<<<tk_grid, kTopkWarps * 32, tk_smem, st>>>(a.logits, a.alpha, a.bt, a.n_experts,
                                                        a.top_k, a.idx, a.w);
  const int nblk = (a.bt + kSegTokens - 1) / kSegTokens;
  const size_t seg_smem = (size_t)kSegWarps * a.n_experts * sizeof(uint32_t);
  seg_count_kernel<<<nblk, kSegThreads, seg_smem, st>>>(a.idx, a.bt, a.top_k, a.n_experts,
                                                        a.block_cnt);
  seg_scan_kernel<<<1, 1024, 2 * a.n_experts * sizeof(int32_t), st>>>(
      a.block_cnt, nblk, a.n_experts, a.tile_m, a.counts, a.offsets, a.mtile_off, a.user_counts);
  seg_scatter_kernel<<<nblk, kSegThreads, seg_smem, st>>>(a.idx, a.bt, a.top_k, a.n_experts,
                                                          a.block_cnt, a.perm, a.inv);
  return cudaGetLastError();
}

cudaError_t launch_segments(const int32_t* idx, int bt, int top_k, int n_experts, int32_t* block_cnt,
                            int32_t* counts, int32_t* offsets, int32_t* mtile_off, int32_t* perm, int32_t* inv,
                            int32_t* user_counts, cudaStream_t st) {
  if (bt <= 0) return cudaSuccess;
  const int nblk = (bt + kSegTokens - 1) / kSegTokens;
  const size_t seg_smem = (size_t)kSegWarps * n_experts * sizeof(uint32_t);
  seg_count_kernel<<<nblk, kSegThreads, seg_smem, st>>>(idx, bt, top_k, n_experts, block_cnt);
  seg_scan_kernel<<<1, 1024, 2 * n_experts * sizeof(int32_t), st>>>(block_cnt, nblk, n_experts, kTileM, counts,
                                                                    offsets, mtile_off, user_counts);
  seg_scatter_kernel<<<nblk, kSegThreads, seg_smem, st>>>(idx, bt, top_k, n_experts, block_cnt, perm, inv);
  return cudaGetLastError();
}

cudaError_t route_tail_prepare() {
  // dynamic shared memory above 48 KB for the largest supported expert count
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)topk_smem_bytes(kMaxExperts));
  if (e != cudaSuccess) return e;
  const int seg = kSegWarps * kMaxExperts * (int)sizeof(uint32_t);
  e = cudaFuncSetAttribute(seg_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, seg);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(seg_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, seg);
}

}  // namespace lmoe
