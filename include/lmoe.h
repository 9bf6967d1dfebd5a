/*
 * lmoe.h -- C ABI of the Stable LatentMoE layer forward for one B300 (sm_103a).
 *
 * The layer ("KimiK3的StableLatentMoE架构解析", tech.news18a.com: ¶"从代码结构看" / Fig. 1 lists
 * router, down_proj, experts, latent_norm, up_proj and shared; ¶"具体前向流程" / Fig. 2 gives
 * the order), for a flattened batch x[bt, d]:
 *
 *   l      = x W_r^T (+ b)                      router logits, fp32          [bt, E]
 *   s      = sigmoid(l)                                                       (fp64)
 *   alpha_e = quantile_{1-K/E}(s[:, e])          Quantile Balancing cutoff    [E]   (fp64)
 *   idx[t] = top-K of (s[t, :] - alpha), ties to the lower expert index, key-descending
 *   w[t,k] = s[t, idx[t,k]] / sum_k' s[t, idx[t,k']]
 *   z      = x W_down^T                          d -> latent
 *   y_tk   = W_d[e] act(W_g[e] z_t, W_u[e] z_t)  e = idx[t,k]   (GroupedExperts, latent width)
 *   c_t    = sum_k w[t,k] * gamma * y_tk / sqrt(mean(y_tk^2) + eps)   (latent_norm, weighted fusion)
 *   out_t  = W_up c_t + sum_j W_d^sh[j] act(W_g^sh[j] x_t, W_u^sh[j] x_t)  (up_proj + 2 shared)
 *
 *   act(g, u) = g' sigmoid(g') u',  g' = beta tanh(g / beta),  u' = beta_u tanh(u / beta_u)
 *   (SiTU-GLU, same page ¶"第一"; beta = 4, beta_u = 25).
 *
 * Shapes at the pages' size ("Vue d'ensemble de l'architecture", mkdocs.reaper.mx, sections
 * "Le budget de paramètres" and "Par où l'information passe"): d = 7168, latent = 3584,
 * E = 896, K = 16, 2 shared experts, intermediate 3072.
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers on the current CUDA device, row-major, densely
 *     packed, 16-byte aligned.  Weights are [out, in] (nn.Linear layout), so both GEMM
 *     operands are K-major.  Element type = cfg.dtype (fp32 or bf16) unless stated.
 *   - The caller owns x, out, every weight and every optional output buffer.  Weights are
 *     borrowed: they are not copied and must stay valid and unchanged while the context
 *     lives.  The context owns its workspace (allocated once, at create, for max_bt tokens).
 *   - Calls are asynchronous and ordered on the given stream (a cudaStream_t; NULL = the
 *     legacy default stream).  A context is used by one stream at a time; calls on two
 *     streams that overlap race on the workspace.
 *   - Errors are returned, never raised or printed: argument errors are found on the host
 *     before any launch and nothing is launched; CUDA runtime errors map to LMOE_ERR_CUDA.
 *     Kernels never trap: a device-side wait that runs out of time or an internal
 *     inconsistency sets a status word that lmoe_sync_status() returns as
 *     LMOE_ERR_TIMEOUT / LMOE_ERR_DEVICE_ASSERT.  With LMOE_CHECK=1 in the environment each
 *     call synchronises its stream and returns that status itself.
 *   - bt == 0 is valid and does nothing; bt > max_bt is LMOE_ERR_INVALID_ARG.
 *   - Non-finite inputs give unspecified (but memory-safe) results.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stdint.h>

#if defined(__GNUC__)
#define LMOE_API __attribute__((visibility("default")))
#else
#define LMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMOE_OK = 0,
  LMOE_ERR_INVALID_ARG = 1,   /* NULL / misaligned / host pointer, bad size, bt > max_bt       */
  LMOE_ERR_UNSUPPORTED = 2,   /* valid layer, but outside what the kernels implement (below)  */
  LMOE_ERR_OOM = 3,           /* workspace allocation failed at create                        */
  LMOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed                          */
  LMOE_ERR_TIMEOUT = 5,       /* a device-side bounded wait expired (kernel returned early)   */
  LMOE_ERR_DEVICE_ASSERT = 6  /* a device-side consistency check failed                       */
} lmoe_status;

typedef enum { LMOE_F32 = 0, LMOE_BF16 = 1 } lmoe_dtype;

/* Layer hyper-parameters.
 * Supported: 1 <= top_k <= n_experts <= 4096, top_k <= 64, 1 <= n_shared <= 3.
 * LMOE_BF16: d, latent, expert_inter, shared_inter multiples of 64 (tensor-core tiles).
 * LMOE_F32 : latent a multiple of 4 (the fp32 path runs on CUDA cores, fp32 FMA).
 * beta, beta_u > 0; rms_eps >= 0.  Anything else: LMOE_ERR_UNSUPPORTED / INVALID_ARG. */
typedef struct {
  int32_t d;             /* model width                                   (7168) */
  int32_t latent;        /* latent width of the routed path               (3584) */
  int32_t n_experts;     /* E, routed experts                             (896)  */
  int32_t top_k;         /* K, experts per token                          (16)   */
  int32_t expert_inter;  /* I, routed expert intermediate size            (3072) */
  int32_t n_shared;      /* S, always-active shared experts               (2)    */
  int32_t shared_inter;  /* Is, shared expert intermediate size           (3072) */
  float beta;            /* SiTU-GLU gate bound                           (4)    */
  float beta_u;          /* SiTU-GLU up-branch bound                      (25)   */
  float rms_eps;         /* latent RMSNorm epsilon                        (1e-6) */
  int32_t dtype;         /* lmoe_dtype of x, out and every weight               */
} lmoe_config;

/* Borrowed weight tensors (device pointers, dtype = cfg.dtype, row-major [out, in]). */
typedef struct {
  const void* w_router;      /* [E, d]                                                   */
  const float* router_bias;  /* [E] fp32, added to the fp32 logits before sigmoid; NULL = none */
  const void* w_down;        /* [latent, d]           W_down                              */
  const void* latent_gamma;  /* [latent]              RMSNorm gain                        */
  const void* w_up;          /* [d, latent]           W_up                                */
  const void* exp_gate;      /* [E, I, latent]        routed expert gate                  */
  const void* exp_up;        /* [E, I, latent]        routed expert up                    */
  const void* exp_down;      /* [E, latent, I]        routed expert down                  */
  const void* sh_gate;       /* [S, Is, d]            shared expert gate                  */
  const void* sh_up;         /* [S, Is, d]            shared expert up                    */
  const void* sh_down;       /* [S, d, Is]            shared expert down                  */
} lmoe_weights;

typedef struct lmoe_ctx lmoe_ctx;
typedef void* lmoe_stream; /* a cudaStream_t */

/* Validate cfg and weights, build the tensor-memory descriptors for the borrowed weights and
 * allocate the workspace for up to max_bt tokens (about bt*K*(I + 2*latent)*2 bytes plus
 * O(bt*(E + d)) for bf16, and 256 KB per SM of fp32 partial sums for the dense GEMMs that
 * small batches split along K) on the current device.  Launches nothing; `stream` is only
 * recorded as the context's default.  On success *out owns the context (free with
 * lmoe_destroy); on any error *out is set to NULL and nothing stays allocated. */
LMOE_API lmoe_status lmoe_create(const lmoe_config* cfg, const lmoe_weights* w, int32_t max_bt,
                        lmoe_stream stream, lmoe_ctx** out);

/* The router alone ("QuantileBalancingRouter", ¶"具体前向流程" and ¶"第三" of the news18a
 * page): logits, sigmoid scores, per-expert cutoffs, top-K, combine weights, per-expert
 * counts and the per-expert token segments (kept in the workspace for lmoe_forward).
 * x: [bt, d].  Every output pointer is an optional device buffer (NULL = not written):
 *   topk_idx      [bt, K] int32   expert ids, key-descending, ties to the lower id
 *   topk_w        [bt, K] fp32    combine weights (sum to 1 per token)
 *   expert_counts [E]     int32   tokens per expert (sum = bt * K)
 *   alpha         [E]     fp64    cutoffs
 *   logits        [bt, E] fp32    router logits including router_bias
 * Outputs are written in stream order; read them after synchronising the stream. */
LMOE_API lmoe_status lmoe_route(lmoe_ctx* ctx, const void* x, int32_t bt, lmoe_stream stream,
                       int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                       double* alpha, float* logits);

/* The whole layer: out[bt, d] (dtype = cfg.dtype) = routed path + shared path for x[bt, d].
 * The cutoffs are computed over the bt tokens of this call (no state across calls, so a
 * batch split into several calls routes differently).  out must not overlap x. */
LMOE_API lmoe_status lmoe_forward(lmoe_ctx* ctx, const void* x, int32_t bt, void* out, lmoe_stream stream);

/* Synchronise `stream`, then return (and clear) the device status word of the context:
 * LMOE_OK, LMOE_ERR_TIMEOUT or LMOE_ERR_DEVICE_ASSERT.
 * Environment: LMOE_CHECK=1 at lmoe_create makes every call of the context synchronise and
 * return this status, and validates the routing index buffers before they are used (see
 * lmoe_debug_check_segments); LMOE_LOG=1 prints one line on stderr for every failing call of
 * this API.  Each lmoe_forward is annotated with NVTX ranges ("lmoe_forward" and one per
 * stage, named as the stages of lmoe_profile) for profilers. */
LMOE_API lmoe_status lmoe_sync_status(lmoe_ctx* ctx, lmoe_stream stream);

/* lmoe_forward with the input and output in host memory: x_host [bt, d] and out_host [bt, d],
 * both of cfg.dtype, page-locked (cudaHostAlloc / cudaHostRegister) for copies that overlap
 * the GPU's work, or pageable (then each copy also stalls the calling thread).  The context
 * stages them through device buffers it owns (two inputs and two outputs of max_bt x d
 * elements, allocated by the first call, which therefore synchronises the device and cannot be
 * captured in a CUDA graph).  The input copy, the forward and the output copy each run on an
 * internal stream of the context, so in a sequence of calls the input copy of the next call and
 * the output copy of the previous one overlap the current forward.  `stream` waits for this
 * call's output copy: out_host is written when `stream` passes the call.  The call does not
 * wait for earlier work on `stream` (its inputs are host memory), except for this context's own
 * device-buffer calls, which are ordered with its forwards internally (they share the context's
 * workspace).  x_host is read at some point after the call is made, so it must already hold the
 * input and stay unchanged until `stream` passes the call.  Errors: as lmoe_forward;
 * LMOE_ERR_INVALID_ARG also for device or managed pointers and overlapping x_host / out_host;
 * LMOE_ERR_OOM if the staging buffers cannot be allocated. */
LMOE_API lmoe_status lmoe_forward_host(lmoe_ctx* ctx, const void* x_host, int32_t bt, void* out_host,
                                       lmoe_stream stream);

/* Synchronise the context's work, free its workspace and the context.  NULL is a no-op. */
LMOE_API void lmoe_destroy(lmoe_ctx* ctx);

/* Static, NUL-terminated name of a status code. */
LMOE_API const char* lmoe_status_string(lmoe_status s);

/* Read-only device pointers to the intermediates of the last route/forward call, for
 * inspection and tests (valid until the next call or lmoe_destroy):
 *   logits [bt, E] fp32, alpha [E] fp64, topk_idx/topk_w [bt, K], offsets [E + 1] int32
 *   (expert segment starts in slot space), perm [bt*K] int32 (slot -> token),
 *   inv [bt, K] int32 ((t, k) -> slot), z [bt, latent], h [bt*K, I] (slot-ordered expert
 *   activations), y [bt*K, latent] (slot-ordered expert outputs), cat [bt, latent + S*Is]
 *   (columns [0, latent) = c, then the S shared activations).  z, h, y, cat are cfg.dtype. */
typedef struct {
  int32_t bt;
  const float* logits;
  const double* alpha;
  const int32_t* topk_idx;
  const float* topk_w;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* inv;
  const void* z;
  const void* h;
  const void* y;
  const void* cat;
} lmoe_workspace_view;

LMOE_API lmoe_status lmoe_workspace(const lmoe_ctx* ctx, lmoe_workspace_view* out);

/* Streaming cutoffs: a variant of the per-call cutoff for callers that route a stream of
 * batches ("KimiK3的StableLatentMoE架构解析", ¶"第三": alpha is adjusted dynamically so each
 * expert's count approaches its quantile target).  With momentum m in [0, 1), every
 * lmoe_route / lmoe_forward on this context uses
 *     alpha = m * alpha_prev + (1 - m) * alpha_batch      (fp64, each step rounded)
 * where alpha_batch is the call's own quantile cutoff and alpha_prev the cutoff the
 * previous call on this context used; the first call after this function uses
 * alpha_batch.  m = 0 (the default) gives per-call cutoffs.  The state lives in the
 * context's workspace and follows stream order.  Returns LMOE_ERR_INVALID_ARG for a NULL
 * context or m outside [0, 1); no GPU work. */
LMOE_API lmoe_status lmoe_set_cutoff_momentum(lmoe_ctx* ctx, double momentum);

/* Placement of the latent RMSNorm.  LMOE_NORM_PER_EXPERT (the default) normalises each
 * (token, expert) latent output before the weighted fusion ("KimiK3的StableLatentMoE架构解析",
 * ¶"具体前向流程" and ¶"第二"):  c = sum_k w_k * gamma * y_k / rms(y_k).
 * LMOE_NORM_COMBINED normalises the weighted sum once, in front of W_up ("Vue d'ensemble de
 * l'architecture", "Par où l'information passe, pour un seul jeton", step f "RMSNorm + W_up"):
 *     c = gamma * s / rms(s),  s = sum_k w_k * y_k,  rms(v) = sqrt(mean(v^2) + rms_eps).
 * Applies to every later lmoe_forward on this context (bf16, fp32, fp8- and MXFP4-expert layers).
 * Returns LMOE_ERR_INVALID_ARG for a NULL context or an unknown placement,
 * LMOE_ERR_UNSUPPORTED for LMOE_NORM_COMBINED with latent > 49152, LMOE_ERR_CUDA if the
 * combine kernel's shared memory limit cannot be raised on the current device.  No GPU
 * work is enqueued. */
typedef enum { LMOE_NORM_PER_EXPERT = 0, LMOE_NORM_COMBINED = 1 } lmoe_latent_norm;
LMOE_API lmoe_status lmoe_set_latent_norm(lmoe_ctx* ctx, lmoe_latent_norm placement);

/* Failure-detection test hook.  Arms the next lmoe_forward on this context so that its
 * routed-expert gate/up kernel leaves its token stages unfilled and limits its device-side
 * waits to 20 ms: the waits run out, the kernel records the timeout in the status word,
 * finishes its in-flight copies and matrix operations, frees its tensor memory and returns
 * (no trap, no hang).  That forward's output is unspecified; lmoe_sync_status then returns
 * LMOE_ERR_TIMEOUT (and clears it) and later calls work normally.  LMOE_ERR_UNSUPPORTED on the
 * CUDA-core engine (fp32 layers). */
LMOE_API lmoe_status lmoe_debug_inject_wait_timeout(lmoe_ctx* ctx);

/* Check of the routing index buffers (the same check LMOE_CHECK=1 runs inside every
 * lmoe_route / lmoe_forward before any kernel indexes memory through them): on the last bt
 * tokens routed on this context, every expert id is in [0, n_experts) and a token's K ids are
 * distinct, the offsets start at 0 and end at bt*K with counts[e] = offsets[e+1] - offsets[e],
 * and every (t, k) slot lies in its expert's segment with perm[slot] = t, so the segments are
 * a permutation of the bt*K (token, k) pairs.  Synchronises `stream`; returns LMOE_OK,
 * LMOE_ERR_DEVICE_ASSERT if a check failed (the status word is cleared), LMOE_OK if nothing
 * has been routed yet. */
LMOE_API lmoe_status lmoe_debug_check_segments(lmoe_ctx* ctx, lmoe_stream stream);

/* Failure-injection test hook on the host: the next device allocation the library makes for a
 * context workspace (lmoe_create, lmoe_create_fp8, lmoe_create_mxfp4) or for lmoe_forward_host's staging buffers
 * fails, and that call returns LMOE_ERR_OOM with nothing leaked.  Process-wide, one shot. */
LMOE_API void lmoe_debug_fail_next_alloc(void);

/* Per-stage device timing.  lmoe_profile(ctx, 1) clears the record and starts recording
 * CUDA events on the call's stream at every stage boundary of each lmoe_forward (up to
 * 1024 calls); lmoe_profile(ctx, 0) stops.  lmoe_profile_read synchronises on the
 * recorded events and writes, per stage, the summed device milliseconds over the recorded
 * calls into ms[LMOE_NUM_STAGES], the number of recorded calls into *calls and the number
 * of kernels those calls launched into *launches (any output may be NULL). */
#define LMOE_NUM_STAGES 9
/* stage order: router GEMM, cutoff + top-K + segments, W_down GEMM, routed token rows into slot
 * order (gather; e4m3 quantization too with fp8 or MXFP4 experts), expert gate/up GEMM, expert down GEMM,
 * RMSNorm + combine, shared gate/up GEMM, W_up + shared-down GEMM */
LMOE_API lmoe_status lmoe_profile(lmoe_ctx* ctx, int32_t enable);
LMOE_API lmoe_status lmoe_profile_read(lmoe_ctx* ctx, float* ms, int32_t* calls, int64_t* launches);

/* Expert segments from given top-K ids, with no allocation by the library.
 * The paper has no counterpart: this is a service to callers that cannot let a library
 * call cudaMalloc, because their device memory belongs to another allocator (such as a
 * framework's caching pool that has reserved the free HBM) or because cudaMalloc's
 * implicit device synchronisation is not acceptable on their path.
 * Computes exactly what lmoe_route leaves in its workspace: a stable counting sort of the
 * bt*top_k (token, k) pairs of topk_idx [bt, top_k] (device, int32, ids in [0, n_experts))
 * by expert, writing expert_counts [n_experts], offsets [n_experts + 1], perm [bt*top_k]
 * (slot -> token) and inv [bt*top_k] ((t, k) -> slot), all caller-owned device buffers.
 * Working memory is one fixed 4 MiB device array inside the library (held on every GPU
 * that loads it until exit), so calls need
 *   (ceil(bt / 128) * n_experts + 2 * n_experts + 1) * 4 bytes <= 4 MiB
 * (e.g. bt <= 149,000 at n_experts = 896); larger calls return LMOE_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (once per device, with
 * that device current); make that first call before any stream capture.  After a device
 * reset (a new primary context) the next call looks it up again.
 * Ids outside [0, n_experts) are a precondition violation that is not reported: such a
 * pair is counted in no segment, so offsets[n_experts] is below bt*top_k, the tail of perm
 * past offsets[n_experts] and the inv entries of those pairs are left unwritten.
 * All calls share the array and it keeps the last call's contents: calls that overlap on
 * the GPU (different streams, or different host threads, without ordering) race on it.
 * bt == 0 returns LMOE_OK without launching. */
LMOE_API lmoe_status lmoe_segments_noalloc(const int32_t* topk_idx, int32_t bt, int32_t top_k,
                                           int32_t n_experts, int32_t* expert_counts, int32_t* offsets,
                                           int32_t* perm, int32_t* inv, lmoe_stream stream);

/* ---------------------------------------------------------------------------------------
 * fp8 (e4m3) routed experts ("KimiK3的StableLatentMoE架构解析", ¶"第一": the bounded SiTU-GLU
 * output is what makes fp8 inference possible).  The routed experts' weights are e4m3 with
 * one fp32 scale per output row; the experts' input z is quantized per token and their
 * activation with one fixed scale from the SiTU-GLU bound (|act| < beta * beta_u):
 *   row quantization: s = absmax / 448 (fp32; 1 for an all-zero row), q = e4m3(x * (1 / s)),
 *                     e4m3 rounding to nearest, ties to even, saturating at +-448;
 *   activation:       q = e4m3(act * (448 / (beta * beta_u))).
 * Router, W_down, W_up and the shared experts stay bf16; the expert GEMMs run as tcgen05
 * kind::f8f6f4 (e4m3 x e4m3 -> fp32).
 * --------------------------------------------------------------------------------------- */
typedef struct {
  const void* exp_gate;      /* e4m3 bytes [E, I, L] (16-byte aligned)                      */
  const void* exp_up;        /* e4m3 bytes [E, I, L]                                         */
  const void* exp_down;      /* e4m3 bytes [E, L, I]                                         */
  const float* gate_scale;   /* [E * I] fp32 row scales of exp_gate                          */
  const float* up_scale;     /* [E * I]                                                      */
  const float* down_scale;   /* [E * L]                                                      */
} lmoe_fp8_experts;

/* As lmoe_create (cfg->dtype must be LMOE_BF16), with the routed experts taken from
 * `experts` (borrowed device buffers, as produced by lmoe_quantize_fp8_rows); w's exp_gate,
 * exp_up and exp_down are not used and may be NULL.  lmoe_route / lmoe_forward /
 * lmoe_destroy work unchanged; in lmoe_workspace's view, h holds the e4m3 activations
 * (bytes).  LMOE_ERR_UNSUPPORTED if the tensor-core engine is disabled (LMOE_FORCE_SIMT). */
LMOE_API lmoe_status lmoe_create_fp8(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_fp8_experts* experts,
                                     int32_t max_bt, lmoe_stream stream, lmoe_ctx** out);

/* Row quantization to e4m3 as described above: w [rows, cols] bf16 (device, 16-byte
 * aligned, cols a multiple of 8) -> q [rows, cols] e4m3 bytes (8-byte aligned) and
 * scale [rows] fp32, on `stream`.  rows == 0 does nothing; bad pointers or sizes give
 * LMOE_ERR_INVALID_ARG, cols not a multiple of 8 LMOE_ERR_UNSUPPORTED.  Expert weights
 * [E, R, C] are quantized as E * R rows of C. */
LMOE_API lmoe_status lmoe_quantize_fp8_rows(const void* w, int64_t rows, int32_t cols, void* q, float* scale,
                                            lmoe_stream stream);

/* ---------------------------------------------------------------------------------------
 * MXFP4 routed experts ("Sparse by design", bittide.aicompass.dev translation of
 * akashbajwa.co: the released model's weights are about 1.4 TB in MXFP4;
 * "KimiK3的StableLatentMoE架构解析", ¶"第一": the bounded SiTU-GLU makes low-precision
 * inference safe).  The format is the OCP microscaling FP4 one: each weight row is cut into
 * blocks of 32 values along its input axis; a block shares a power-of-two scale 2^x stored as
 * the byte x + 127 (ue8m0), x = floor(log2(max |w| of the block)) - 2 clamped to [-127, 127]
 * (-127 for an all-zero block); each value is e2m1(w / 2^x) (magnitudes 0, 0.5, 1, 1.5, 2, 3,
 * 4, 6; nearest, ties to the even mantissa, saturating at 6).  The experts' input z and their
 * activation are e4m3 as for lmoe_create_fp8; router, W_down, W_up and the shared experts stay
 * bf16.  The expert GEMMs run as tcgen05 kind::mxf8f6f4 with block scaling (e2m1 weights x
 * e4m3 tokens -> fp32).
 *
 * Layouts (both written by lmoe_quantize_mxfp4_rows):
 *   codes: [rows, cols / 2] bytes, value 2j of a row in the low nibble of byte j, 2j + 1 in the
 *          high nibble;
 *   scales: tiled in 512-byte groups, one per (128-row block rb, 128-column block kb) at byte
 *          (rb * (cols / 128) + kb) * 512; inside it, the scale of row r (r % 128 = 32 i + l)
 *          for the 32 columns kb * 128 + 32 j ... + 31 is at byte 16 l + 4 i + j.
 * Expert tensors [E, R, C] are E * R rows of C.
 * --------------------------------------------------------------------------------------- */
typedef struct {
  const void* exp_gate;      /* e2m1 codes [E, I, L / 2] bytes (32-byte aligned)             */
  const void* exp_up;        /* e2m1 codes [E, I, L / 2]                                     */
  const void* exp_down;      /* e2m1 codes [E, L, I / 2]                                     */
  const void* gate_sf;       /* ue8m0 block scales of exp_gate, E * I * L / 32 bytes, tiled  */
  const void* up_sf;         /*                    of exp_up                                 */
  const void* down_sf;       /*                    of exp_down, E * L * I / 32 bytes         */
} lmoe_mxfp4_experts;

/* As lmoe_create_fp8, with MXFP4 routed experts (borrowed device buffers, as produced by
 * lmoe_quantize_mxfp4_rows; codes 32-byte and scales 16-byte aligned).  latent and
 * expert_inter must be multiples of 128 (else LMOE_ERR_UNSUPPORTED).  In lmoe_workspace's
 * view, h holds the e4m3 activations (bytes). */
LMOE_API lmoe_status lmoe_create_mxfp4(const lmoe_config* cfg, const lmoe_weights* w,
                                       const lmoe_mxfp4_experts* experts, int32_t max_bt, lmoe_stream stream,
                                       lmoe_ctx** out);

/* MXFP4 quantization as described above: w [rows, cols] bf16 (device, 16-byte aligned) ->
 * codes [rows, cols / 2] bytes (16-byte aligned) and the tiled scales (rows * cols / 32 bytes),
 * on `stream`.  rows == 0 does nothing; negative sizes or NULL / misaligned pointers give
 * LMOE_ERR_INVALID_ARG; rows or cols not a multiple of 128 LMOE_ERR_UNSUPPORTED. */
LMOE_API lmoe_status lmoe_quantize_mxfp4_rows(const void* w, int64_t rows, int32_t cols, void* q, void* sf,
                                              lmoe_stream stream);

/* ---------------------------------------------------------------------------------------
 * Dense SiTU-GLU FFN: the full-width feed-forward block of the model's first (dense) layer
 * ("Vue d'ensemble de l'architecture", mkdocs.reaper.mx, table "Le budget de paramètres,
 * module par module": 727 M parameters, intermediate 33 792 at d = 7168), with the experts'
 * activation ("KimiK3的StableLatentMoE架构解析", ¶"第一"):
 *   out[t] = W_down act(W_gate x[t], W_up x[t]),  act as for the layer above.
 * bf16 only, on the tensor-core engine; d and inter multiples of 64.
 * --------------------------------------------------------------------------------------- */
typedef struct {
  int32_t d;        /* model width                          (7168)  */
  int32_t inter;    /* intermediate width                   (33792) */
  float beta;       /* SiTU-GLU gate bound                  (4)     */
  float beta_u;     /* SiTU-GLU up bound                    (25)    */
} lmoe_ffn_config;

typedef struct lmoe_ffn lmoe_ffn;

/* Borrows w_gate [inter, d], w_up [inter, d], w_down [d, inter] (bf16, device, 16-byte
 * aligned; they must outlive the context) and allocates an activation buffer of
 * max_bt * inter bf16.  Errors as for lmoe_create (INVALID_ARG: bad sizes or pointers;
 * UNSUPPORTED: d or inter not a multiple of 64; OOM; CUDA). */
LMOE_API lmoe_status lmoe_ffn_create(const lmoe_ffn_config* cfg, const void* w_gate, const void* w_up,
                                     const void* w_down, int32_t max_bt, lmoe_ffn** out);
/* out [bt, d] bf16 = the FFN of x [bt, d] bf16, on `stream` (asynchronous; two kernels).
 * bt == 0 does nothing; bt > max_bt, NULL or misaligned pointers, or out overlapping x
 * give LMOE_ERR_INVALID_ARG.  A context is used by one stream at a time. */
LMOE_API lmoe_status lmoe_ffn_forward(lmoe_ffn* ffn, const void* x, int32_t bt, void* out, lmoe_stream stream);
/* Synchronises `stream` and returns (then clears) the device status of this context's
 * kernels (LMOE_ERR_TIMEOUT when a bounded device-side wait ran out). */
LMOE_API lmoe_status lmoe_ffn_sync_status(lmoe_ffn* ffn, lmoe_stream stream);
/* NULL-safe; synchronises the device, frees the activation buffer. */
LMOE_API void lmoe_ffn_destroy(lmoe_ffn* ffn);

/* Library build identifier (static string): engine names per dtype. */
LMOE_API const char* lmoe_build_info(void);

#ifdef __cplusplus
}
#endif
#endif /* LMOE_H */
