// CUDA-core GEMM with fp32 FMA accumulation: the engine of the fp32 layer (tensor-core
// fp32 modes round operands to tf32, which the fp32 tolerance does not allow).  It runs
// every contraction of the layer: router logits (+ transposed copy), W_down, the grouped
// routed experts with the row gather and the SiTU-GLU epilogue, the shared experts and
// the K-concatenated W_up / shared-down projection.
#include "common.cuh"
#include "internal.h"

namespace lmoe {

constexpr int kSBM = 128, kSBN = 64, kSBK = 16, kSThreads = 256;

template <typename T>
__device__ __forceinline__ float load_b(const GemmArgs& a, int g, int n, int k) {
  int s = 0;
#pragma unroll
  for (int i = 1; i < kMaxKSeg; ++i)
    if (i < a.nseg && k >= a.seg_k0[i]) s = i;
  const T* B = static_cast<const T*>(a.seg_B[s]);
  long long row = a.seg_row0[s] + (long long)g * a.b_group_rows + n;
  return to_f(B[row * a.seg_ldb[s] + (k - a.seg_k0[s])]);
}

template <typename T, int EPI>
__global__ void __launch_bounds__(kSThreads)
gemm_simt_kernel(const GemmArgs a) {
  __shared__ float As[kSBK][kSBM];
  __shared__ float Bs[kSBK][kSBN];
  __shared__ float Bu[EPI == kEpiGlu ? kSBK : 1][kSBN];

  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * kSBN;
  int g = 0, row0, row_end;
  if (a.seg_off) {
    const int total = a.mtile_off[a.G];
    const int mt = blockIdx.y;
    if (mt >= total) return;
    int lo = 0, hi = a.G;                       // largest g with mtile_off[g] <= mt
    while (hi - lo > 1) { int mid = (lo + hi) >> 1; if (a.mtile_off[mid] <= mt) lo = mid; else hi = mid; }
    g = lo;
    const int tile0 = a.seg_off[g] + (mt - a.mtile_off[g]) * kTileM;   // this m-tile: kTileM rows
    row0 = tile0 + blockIdx.z * kSBM;                                    // at most 2 * kSBM
    row_end = min(a.seg_off[g + 1], tile0 + kTileM);
  } else {
    row0 = blockIdx.y * kSBM;
    row_end = a.M;
  }
  if (row0 >= row_end) return;

  const T* A = static_cast<const T*>(a.A);
  const T* Bup = static_cast<const T*>(a.B_up);
  const int ty = tid >> 4, tx = tid & 15;
  float acc[8][4], accu[EPI == kEpiGlu ? 8 : 1][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc[i][j] = 0.f; if (EPI == kEpiGlu) accu[i][j] = 0.f; }

  // this thread's A row for loading
  const int lr = tid >> 1, lk0 = (tid & 1) * 8;
  const int grow = row0 + lr;
  long long arow = -1;
  if (grow < row_end) arow = a.a_rows ? (long long)a.a_rows[grow] : (long long)grow;
  const int bn = tid >> 2, bk0 = (tid & 3) * 4;

  for (int k0 = 0; k0 < a.K; k0 += kSBK) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int k = k0 + lk0 + i;
      As[lk0 + i][lr] = (arow >= 0 && k < a.K) ? to_f(A[arow * a.lda + k]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int k = k0 + bk0 + i, n = n0 + bn;
      bool ok = (k < a.K) && (n < a.N);
      Bs[bk0 + i][bn] = ok ? load_b<T>(a, g, n, k) : 0.f;
      if (EPI == kEpiGlu) {
        long long row = (long long)g * a.b_group_rows + n;
        Bu[bk0 + i][bn] = ok ? to_f(Bup[row * a.seg_ldb[0] + k]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSBK; ++kk) {
      float av[8], bv[4], uv[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) av[i] = As[kk][ty * 8 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) { bv[j] = Bs[kk][tx * 4 + j]; if (EPI == kEpiGlu) uv[j] = Bu[kk][tx * 4 + j]; }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (EPI == kEpiGlu) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = row0 + ty * 8 + i;
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      if (EPI == kEpiStore) {
        static_cast<T*>(a.out)[(long long)r * a.ldo + n] = from_f<T>(acc[i][j]);
      } else if (EPI == kEpiGlu) {
        static_cast<T*>(a.out)[(long long)r * a.ldo + n] =
            from_f<T>(situ_glu(acc[i][j], accu[i][j], a.beta, a.beta_u));
      } else {
        float v = acc[i][j] + (a.bias ? a.bias[n] : 0.f);
        static_cast<float*>(a.out)[(long long)r * a.ldo + n] = v;
        a.out_t[(long long)n * a.ldt + r] = v;
      }
    }
  }
}

template <typename T>
static cudaError_t launch_t(const GemmArgs& a, cudaStream_t st) {
  static_assert(kTileM <= 2 * kSBM, "a grouped m-tile spans at most two CUDA-core row blocks");
  dim3 grid((a.N + kSBN - 1) / kSBN, a.seg_off ? a.max_mtiles : (a.M + kSBM - 1) / kSBM, a.seg_off ? 2 : 1);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  switch (a.epi) {
    case kEpiStore: gemm_simt_kernel<T, kEpiStore><<<grid, kSThreads, 0, st>>>(a); break;
    case kEpiGlu: gemm_simt_kernel<T, kEpiGlu><<<grid, kSThreads, 0, st>>>(a); break;
    default: gemm_simt_kernel<T, kEpiRouter><<<grid, kSThreads, 0, st>>>(a); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_gemm_simt(const GemmArgs& a, bool is_bf16, cudaStream_t st) {
  return is_bf16 ? launch_t<bf16>(a, st) : launch_t<float>(a, st);
}

}  // namespace lmoe
