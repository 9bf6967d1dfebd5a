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
                 double* __restrict__ alpha, const double* __restrict__ alpha_prev, double momentum,
                 double* __restrict__ alpha_state, int32_t* __restrict__ list_count) {
  const int e = blockIdx.x;
  if (e == 0 && threadIdx.x == 0) *list_count = 0;   // the top-K kernels' list starts empty
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
    // streaming variant: a moving average with the previous call's cutoff, evaluated as
    // m * prev + (1 - m) * a, each step rounded (no fused multiply-add)
    if (alpha_prev) a = __dadd_rn(__dmul_rn(momentum, alpha_prev[e]), __dmul_rn(__dsub_rn(1.0, momentum), a));
    alpha[e] = a;
    if (alpha_state) alpha_state[e] = a;
  }
}

// ------------------------------------------------------------------------------------
// Top-K per token: one warp per token, exact in fp64 but with fp64 work only where it can
// change the answer (the fp64 pipe of this GPU is narrow, so the bulk stays in fp32 and
// integer arithmetic).
//   1. fp32 keys k32[e] = 1 / (1 + expf(-l)) - (float)alpha[e] for every expert, kept as
//      order-preserving uint32.  Against the fp64 key s - alpha the error is at most
//      4.5e-7 (expf within 2 ulp; correctly rounded add, divide, conversion and subtract;
//      keys lie in [-1, 1]); kKeyTol = 1e-6 bounds it.
//   2. v = the K-th largest k32, built bit by bit from warp-wide counts (32 steps).
//   3. Any expert with k32 < v - 2 kKeyTol has an fp64 key below the K-th largest fp64 key
//      (K experts have fp64 keys >= v - kKeyTol), so it cannot be chosen: the candidates
//      are the experts with k32 >= v - 2 kKeyTol (usually K or K+1 of them).
//   4. Each candidate's rank among the candidates (key descending, ties to the lower expert
//      index) is its output slot if below K.  Two candidates whose fp32 keys differ by more
//      than 2 kKeyTol compare in fp32 (their fp64 keys are in the same order); closer pairs
//      compare their fp64 keys, which are computed only for candidates with such a
//      neighbour (on this GPU's narrow fp64 pipe the fp64 sigmoid dominated the kernel).
//      With more than 32 candidates (near-ties, K > 32) K rounds of warp argmax over fp64
//      keys do the same.
// Combine weights are the chosen fp64 scores over their sum (summed in k order).
// ------------------------------------------------------------------------------------
constexpr float kKeyTol = 1e-6f;
constexpr double kTaken64 = -3.0;     // below every key (keys lie in [-1, 1])
constexpr int kTopkMaxWarps = 8;
constexpr int kRegKeys = 32;          // keys per lane held in registers (E <= 1024)
constexpr size_t kTopkSmemCap = 96 * 1024;

__device__ __forceinline__ bool topk_better(bool v1, double k1, int e1, bool v2, double k2, int e2) {
  if (v1 != v2) return v1;
  if (!v1) return false;
  return k1 > k2 || (k1 == k2 && e1 < e2);
}

// Warp argmax over lane-held (valid, key, index); ties to the lower index.  All lanes get
// the winner.
__device__ __forceinline__ void warp_best(bool& v, double& k, int& e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const bool v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const double k2 = __shfl_xor_sync(0xffffffffu, k, o);
    const int e2 = __shfl_xor_sync(0xffffffffu, e, o);
    if (topk_better(v2, k2, e2, v, k, e)) { v = v2; k = k2; e = e2; }
  }
}

__global__ void __launch_bounds__(kTopkMaxWarps * 32)
topk_kernel(const float* __restrict__ logits, const double* __restrict__ alpha, int bt,
            int n_experts, int top_k, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
            const int32_t* __restrict__ list, const int32_t* __restrict__ list_count) {
  extern __shared__ double smem_d[];
  const int nwarps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = n_experts;
  double* s_alpha = smem_d;                                                       // [E]
  double* ckey = smem_d + E + (size_t)warp * E;                                   // [E] candidate fp64 keys
  double* chosen_s = smem_d + (size_t)(nwarps + 1) * E + (size_t)warp * kMaxTopK; // [K]
  float* s_alpha32 = reinterpret_cast<float*>(smem_d + (size_t)(nwarps + 1) * E + (size_t)nwarps * kMaxTopK);
  uint32_t* ku = reinterpret_cast<uint32_t*>(s_alpha32 + E) + (size_t)warp * 2 * E;   // [E] fp32 keys
  int32_t* cid = reinterpret_cast<int32_t*>(ku + E);                              // [E] candidates
  if (list && *list_count == 0) return;

  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double a = alpha[e];
    s_alpha[e] = a;
    s_alpha32[e] = (float)a;
  }
  __syncthreads();

  // every token, or only the tokens of the list (those the fast kernel left to this one)
  const int ntok = list ? *list_count : bt;
  for (int it = blockIdx.x * nwarps + warp; it < ntok; it += gridDim.x * nwarps) {
    const int t = list ? list[it] : it;
    const float* lrow = logits + (size_t)t * E;
    // 1. fp32 keys (also kept in registers when every lane has at most kRegKeys of them)
    uint32_t kr[kRegKeys];
    if (E <= 32 * kRegKeys) {
#pragma unroll
      for (int i = 0; i < kRegKeys; ++i) {
        const int e = lane + 32 * i;
        kr[i] = 0u;
        if (e < E) {
          kr[i] = f32_to_key(1.0f / (1.0f + expf(-lrow[e])) - s_alpha32[e]);
          ku[e] = kr[i];
        }
      }
    } else {
      for (int e = lane; e < E; e += 32) ku[e] = f32_to_key(1.0f / (1.0f + expf(-lrow[e])) - s_alpha32[e]);
    }
    __syncwarp();
    // 2. the K-th largest key: the largest v with at least K keys >= v (key 0 is below every
    //    real key, so the register slots past E never count)
    uint32_t v = 0;
    if (E <= 32 * kRegKeys) {
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = v | (1u << bit);
        uint32_t c = 0;
#pragma unroll
        for (int i = 0; i < kRegKeys; ++i) c += kr[i] >= cand ? 1u : 0u;
        if (__reduce_add_sync(0xffffffffu, c) >= (uint32_t)top_k) v = cand;
      }
    } else {
      for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = v | (1u << bit);
        uint32_t c = 0;
        for (int e = lane; e < E; e += 32) c += ku[e] >= cand ? 1u : 0u;
        if (__reduce_add_sync(0xffffffffu, c) >= (uint32_t)top_k) v = cand;
      }
    }
    // 3. candidates
    const uint32_t thr = f32_to_key(key_to_f32(v) - 2.0f * kKeyTol);
    int nc = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool c = e < E && ku[e] >= thr;
      const unsigned m = __ballot_sync(0xffffffffu, c);
      if (c) cid[nc + __popc(m & ((1u << lane) - 1u))] = e;
      nc += __popc(m);
    }
    __syncwarp();
    // 4. exact selection among the candidates
    if (nc <= 32) {
      // Two candidates whose fp32 keys differ by more than 2 kKeyTol have their fp64 keys in the
      // same order; only candidates with a neighbour closer than that need their fp64 key, and
      // the fp64 evaluation is skipped when no candidate of the token needs it.
      const int ej = lane < nc ? cid[lane] : 0;
      const float kj32 = lane < nc ? key_to_f32(ku[ej]) : 0.f;
      bool near = false;
      if (lane < nc)
        for (int i = 0; i < nc; ++i)
          if (i != lane && fabsf(key_to_f32(ku[cid[i]]) - kj32) <= 2.0f * kKeyTol) near = true;
      if (__any_sync(0xffffffffu, near)) {
        if (near) ckey[lane] = sigmoid_f64((double)lrow[ej]) - s_alpha[ej];
        __syncwarp();
      }
      if (lane < nc) {
        int rank = 0;
        for (int i = 0; i < nc; ++i) {
          const int ei = cid[i];
          const float ki32 = key_to_f32(ku[ei]);
          bool beats;
          if (fabsf(ki32 - kj32) > 2.0f * kKeyTol) {
            beats = ki32 > kj32;
          } else {
            const double ki = ckey[i], kj = ckey[lane];   // both near: fp64 keys computed above
            beats = ki > kj || (ki == kj && ei < ej);
          }
          rank += (i != lane && beats) ? 1 : 0;
        }
        if (rank < top_k) {
          idx_out[(size_t)t * top_k + rank] = ej;
          chosen_s[rank] = (double)ej;
        }
      }
    } else {
      for (int j = lane; j < nc; j += 32) {
        const int e = cid[j];
        ckey[j] = sigmoid_f64((double)lrow[e]) - s_alpha[e];
      }
      __syncwarp();
      bool bv = false;
      double bk = 0.0;
      int be = 0;
      for (int j = lane; j < nc; j += 32)
        if (topk_better(true, ckey[j], cid[j], bv, bk, be)) { bv = true; bk = ckey[j]; be = cid[j]; }
      for (int k = 0; k < top_k; ++k) {
        bool wv = bv;
        double wk = bk;
        int we = be;
        warp_best(wv, wk, we);
        if (lane == 0) {
          idx_out[(size_t)t * top_k + k] = we;
          chosen_s[k] = (double)we;
        }
        if (bv && be == we) {
          // this lane held the winner (each expert is one candidate): drop it and rescan
          bv = false;
          for (int j = lane; j < nc; j += 32) {
            if (cid[j] == we) ckey[j] = kTaken64;
            const double kd = ckey[j];
            if (kd == kTaken64) continue;
            if (topk_better(true, kd, cid[j], bv, bk, be)) { bv = true; bk = kd; be = cid[j]; }
          }
        }
      }
    }
    __syncwarp();
    // combine weights: chosen raw scores over their sum (summed in k order, fp64)
    for (int k = lane; k < top_k; k += 32) {
      const int e = (int)chosen_s[k];
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

// ------------------------------------------------------------------------------------
// Top-K, fast path (E <= 32 * kRegKeys, K <= 32): one warp per token with the token's fp32
// keys in registers.  A float threshold t with at least K keys >= t and at most 32 keys >=
// t - 2 kKeyTol is found by bisection (keys lie in (-1, 1); the K-th key usually sits near 0,
// where the cutoffs put about K of the E keys above zero).  Every expert below t - 2 kKeyTol
// then has an fp64 key below those of the >= K experts at or above t, so the selection lies
// among the <= 32 candidates, which are ranked exactly as in topk_kernel (fp64 keys only for
// candidates with a neighbour closer than 2 kKeyTol).  Tokens with no such threshold (massive
// ties) are appended to `list` for topk_kernel.  Same outputs as topk_kernel, bit for bit.
// ------------------------------------------------------------------------------------
constexpr int kFastWarps = 8;

__global__ void __launch_bounds__(kFastWarps * 32)
topk_fast_kernel(const float* __restrict__ logits, const double* __restrict__ alpha, int bt, int n_experts,
                 int top_k, int32_t* __restrict__ idx_out, float* __restrict__ w_out, int32_t* __restrict__ list,
                 int32_t* __restrict__ list_count) {
  extern __shared__ double smem_d[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = n_experts;
  double* s_alpha = smem_d;                                                    // [E]
  double* ck64 = smem_d + E + warp * 32;                                       // [32] per warp
  double* chosen_s = smem_d + E + kFastWarps * 32 + warp * 32;                 // [32] per warp
  float* s_alpha32 = reinterpret_cast<float*>(smem_d + E + kFastWarps * 64);   // [E]
  float* ck32 = s_alpha32 + E + warp * 32;                                     // [32] per warp
  int32_t* cid = reinterpret_cast<int32_t*>(s_alpha32 + E + kFastWarps * 32) + warp * 32;  // [32] per warp
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double a = alpha[e];
    s_alpha[e] = a;
    s_alpha32[e] = (float)a;
  }
  __syncthreads();
  const unsigned full = 0xffffffffu;
  const bool usable = E <= 32 * kRegKeys && top_k <= 32;
  for (int t = blockIdx.x * kFastWarps + warp; t < bt; t += gridDim.x * kFastWarps) {
    if (!usable) {
      if (lane == 0) list[atomicAdd(list_count, 1)] = t;
      continue;
    }
    const float* lrow = logits + (size_t)t * E;
    float kf[kRegKeys];
#pragma unroll
    for (int i = 0; i < kRegKeys; ++i) {
      const int e = lane + 32 * i;
      kf[i] = e < E ? 1.0f / (1.0f + expf(-lrow[e])) - s_alpha32[e] : -INFINITY;
    }
    auto count_ge = [&](float thr) {
      uint32_t c = 0;
#pragma unroll
      for (int i = 0; i < kRegKeys; ++i) c += kf[i] >= thr ? 1u : 0u;
      return (int)__reduce_add_sync(full, c);
    };
    // threshold: count(>= t) >= K and count(>= t - 2 tol) <= 32
    float lo = -2.0f, hi = 2.0f, tt = 0.0f;
    bool found = false;
    for (int step = 0; step < 48; ++step) {
      if (count_ge(tt) < top_k) {
        hi = tt;
      } else if (count_ge(tt - 2.0f * kKeyTol) <= 32) {
        found = true;
        break;
      } else {
        lo = tt;
      }
      const float mid = 0.5f * (lo + hi);
      if (mid == lo || mid == hi) break;
      tt = mid;
    }
    if (!found) {
      if (lane == 0) list[atomicAdd(list_count, 1)] = t;
      continue;
    }
    // candidates, in expert order
    const float thr = tt - 2.0f * kKeyTol;
    int nc = 0;
#pragma unroll
    for (int i = 0; i < kRegKeys; ++i) {
      const bool c = kf[i] >= thr;
      const unsigned m = __ballot_sync(full, c);
      if (c) {
        const int pos = nc + __popc(m & ((1u << lane) - 1u));
        cid[pos] = lane + 32 * i;
        ck32[pos] = kf[i];
      }
      nc += __popc(m);
    }
    __syncwarp();
    // exact ranks: fp32 order for candidates further apart than 2 tol, fp64 keys otherwise.
    // Each candidate's fp64 score is computed once (one pass of the narrow fp64 pipe per
    // token) and serves both its fp64 key and, if chosen, its combine weight.
    const int ej = lane < nc ? cid[lane] : 0;
    const float kj32 = lane < nc ? ck32[lane] : 0.f;
    const double sj = lane < nc ? sigmoid_f64((double)lrow[ej]) : 0.0;
    bool near = false;
    if (lane < nc)
      for (int i = 0; i < nc; ++i)
        if (i != lane && fabsf(ck32[i] - kj32) <= 2.0f * kKeyTol) near = true;
    if (__any_sync(full, near)) {
      if (near) ck64[lane] = sj - s_alpha[ej];
      __syncwarp();
    }
    if (lane < nc) {
      int rank = 0;
      for (int i = 0; i < nc; ++i) {
        const float ki32 = ck32[i];
        bool beats;
        if (fabsf(ki32 - kj32) > 2.0f * kKeyTol) {
          beats = ki32 > kj32;
        } else {
          const double ki = ck64[i], kj = ck64[lane];
          beats = ki > kj || (ki == kj && cid[i] < ej);
        }
        rank += (i != lane && beats) ? 1 : 0;
      }
      if (rank < top_k) {
        idx_out[(size_t)t * top_k + rank] = ej;
        chosen_s[rank] = sj;
      }
    }
    __syncwarp();
    // combine weights: chosen raw scores over their sum (summed in k order, fp64)
    double total = 0.0;
    for (int k = 0; k < top_k; ++k) total = total + chosen_s[k];
    if (lane < top_k) w_out[(size_t)t * top_k + lane] = (float)(chosen_s[lane] / total);
    __syncwarp();
  }
}

size_t topk_fast_smem_bytes(int n_experts) {
  return (size_t)n_experts * (sizeof(double) + sizeof(float)) + (size_t)kFastWarps * 32 * (2 * sizeof(double) + sizeof(float) + sizeof(int32_t));
}

size_t topk_smem_bytes(int n_experts, int nwarps) {
  return (size_t)(nwarps + 1) * n_experts * sizeof(double) + (size_t)nwarps * kMaxTopK * sizeof(double) +
         (size_t)n_experts * sizeof(float) + (size_t)nwarps * 2 * n_experts * sizeof(uint32_t);
}

// Warps per block that fit the shared-memory budget (at least one; a single warp may
// exceed the budget slightly at the largest expert count, which the launch attribute allows).
int topk_warps(int n_experts) {
  int w = kTopkMaxWarps;
  while (w > 1 && topk_smem_bytes(n_experts, w) > kTopkSmemCap) --w;
  return w;
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
  qb_cutoff_kernel<<<a.n_experts, kCutoffThreads, 0, st>>>(a.logits_t, a.bt, a.n_experts, a.top_k, a.alpha,
                                                          a.alpha_prev, a.momentum, a.alpha_state, a.list_count);
  const int sms = a.sm_count > 0 ? a.sm_count : 1;
  // fast path for every token it can decide; the exact general kernel for the listed rest
  int fast_grid = (a.bt + kFastWarps - 1) / kFastWarps;
  if (fast_grid > sms * 8) fast_grid = sms * 8;
  topk_fast_kernel<<<fast_grid, kFastWarps * 32, topk_fast_smem_bytes(a.n_experts), st>>>(
      a.logits, a.alpha, a.bt, a.n_experts, a.top_k, a.idx, a.w, a.list, a.list_count);
  const int tk_warps = topk_warps(a.n_experts);
  const size_t tk_smem = topk_smem_bytes(a.n_experts, tk_warps);
  int tk_grid = (a.bt + tk_warps - 1) / tk_warps;
  if (tk_grid > sms * 2) tk_grid = sms * 2;
  topk_kernel<<<tk_grid, tk_warps * 32, tk_smem, st>>>(a.logits, a.alpha, a.bt, a.n_experts,
                                                      a.top_k, a.idx, a.w, a.list, a.list_count);
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
                                       (int)topk_smem_bytes(kMaxExperts, topk_warps(kMaxExperts)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)topk_fast_smem_bytes(kMaxExperts));
  if (e != cudaSuccess) return e;
  const int seg = kSegWarps * kMaxExperts * (int)sizeof(uint32_t);
  e = cudaFuncSetAttribute(seg_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, seg);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(seg_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, seg);
}

}  // namespace lmoe
