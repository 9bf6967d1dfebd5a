// Internal launcher interfaces between the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

constexpr int kMaxExperts = 4096;
constexpr int kMaxTopK = 64;
constexpr int kMaxShared = 3;
constexpr int kSegTokens = 128;   // tokens per block of the segmentation kernels
constexpr int kTileM = 192;       // tokens per grouped GEMM tile (m-tile prefix granularity): CUDA-core
                                  // engine and MXFP4 experts
constexpr int kTileWide = 256;    // tokens per grouped tensor-core tile of the bf16 and e4m3 experts

struct RouteArgs {
  const float* logits;      // [bt, E]
  const float* logits_t;    // [E, bt]
  int bt, n_experts, top_k, tile_m;
  double* alpha;            // [E]
  const double* alpha_prev; // [E] previous call's cutoff (streaming cutoffs), or null
  double momentum;          // weight of alpha_prev
  double* alpha_state;      // [E] where this call's cutoff is kept for the next, or null
  int32_t* idx;             // [bt, K]
  float* w;                 // [bt, K]
  int32_t* block_cnt;       // [ceil(bt / kSegTokens), E]
  int32_t* counts;          // [E]
  int32_t* offsets;         // [E + 1]
  int32_t* mtile_off;       // [E + 1]
  int32_t* perm;            // [bt * K]
  int32_t* inv;             // [bt * K]
  int32_t* user_counts;     // optional [E]
  int sm_count;             // SMs of the device (grid sizing)
  int32_t* list;            // [bt] tokens the fast top-K kernel leaves to the general one
  int32_t* list_count;      // [1]
};

constexpr int kRouteTailLaunches = 6;   // cutoff, top-K (fast, general), count, scan, scatter
cudaError_t route_tail_prepare();
cudaError_t launch_route_tail(const RouteArgs& a, cudaStream_t st);
// Only the segmentation chain (count, scan, scatter) on caller-supplied buffers.
cudaError_t launch_segments(const int32_t* idx, int bt, int top_k, int n_experts, int32_t* block_cnt,
                            int32_t* counts, int32_t* offsets, int32_t* mtile_off, int32_t* perm, int32_t* inv,
                            int32_t* user_counts, cudaStream_t st);

// ---------------------------------------------------------------------------- GEMMs
// C[r, n] = sum_k A[arow(r), k] * B(g, n, k), with
//   arow(r) = a_rows ? a_rows[r] : r            (row gather for the routed experts)
//   B(g, n, k) = seg_B[s][(g * b_group_rows + n) * seg_ldb[s] + (k - seg_k0[s])]
//               for the K segment s holding k    (K-concatenation of several weights)
// Rows are grouped when seg_off != nullptr: group g owns rows [seg_off[g], seg_off[g+1])
// and its m-tiles are numbered from mtile_off[g] (device arrays, set by the router).
enum EpiKind { kEpiStore = 0, kEpiGlu = 1, kEpiRouter = 2 };
// Which contraction of the layer a GemmArgs describes (the tensor-core engine keys its
// prebuilt weight descriptors on it).
enum GemmOp { kOpRouter = 0, kOpDown, kOpExpertGateUp, kOpExpertDown, kOpSharedGateUp, kOpFinal, kNumOps };

constexpr int kMaxKSeg = 1 + kMaxShared;

struct GemmArgs {
  int M, N, K;                   // M: rows (dense), or the row capacity (grouped)
  const void* A; long long lda;
  const int32_t* a_rows;
  int nseg;
  int seg_k0[kMaxKSeg + 1];      // seg_k0[nseg] == K
  const void* seg_B[kMaxKSeg];
  long long seg_ldb[kMaxKSeg];
  long long seg_row0[kMaxKSeg];  // extra B row offset per segment (e.g. shared expert j * d)
  const void* B_up;              // GLU: up-branch weights, same layout as segment 0
  long long b_group_rows;        // grouped: B rows per group (0 = same B for all groups)
  const int32_t* seg_off;        // [G + 1] or nullptr
  const int32_t* mtile_off;      // [G + 1] or nullptr
  int G;
  int bt_tokens;                 // grouped: tokens of the call (rows of A before the gather)
  int max_mtiles;                // launch bound on m-tiles (grouped)
  int epi;
  void* out; long long ldo;      // Store / Glu: T; Router: fp32
  float* out_t; long long ldt;   // Router: transposed logits [N, ldt]
  const float* bias;             // Router: [N] or nullptr
  float beta, beta_u;
  int op;                        // GemmOp
};

cudaError_t launch_gemm_simt(const GemmArgs& a, bool is_bf16, cudaStream_t st);

// fp8 experts: q[r] = e4m3 row r of the bf16 rows x [rows, cols] with its scale (csrc/fp8.cu).
cudaError_t launch_quantize_rows(const void* x, long long rows, int cols, void* q, float* scale, int grid,
                                 cudaStream_t st);

// ---------------------------------------------------------------------------- checks
// Sets kStatusAssert in *status unless idx / counts / offsets / perm / inv form valid
// expert segments of bt*top_k (token, k) pairs (csrc/check.cu).
cudaError_t launch_validate_segments(const int32_t* idx, const int32_t* counts, const int32_t* offsets,
                                     const int32_t* perm, const int32_t* inv, int bt, int top_k, int n_experts,
                                     uint32_t* status, int sm_count, cudaStream_t st);

// ---------------------------------------------------------------------------- combine
struct CombineArgs {
  const void* y;          // [bt*K, L] slot-ordered expert outputs
  const int32_t* inv;     // [bt, K]
  const float* w;         // [bt, K]
  const void* gamma;      // [L]
  int bt, top_k, latent;
  float eps;
  void* cat; long long ldc;   // c written to cat[t, 0:L]
  bool norm_sum;              // RMSNorm of the weighted sum instead of each expert row
};
// Largest latent width the norm-on-sum combine supports (its fp32 row lives in shared memory).
constexpr int kMaxNormSumLatent = 48 * 1024;
// Raises the combine kernel's dynamic shared memory limit for norm_sum at this latent width.
cudaError_t prepare_combine(int latent, bool norm_sum);
cudaError_t launch_combine(const CombineArgs& a, bool is_bf16, cudaStream_t st);

}  // namespace lmoe
