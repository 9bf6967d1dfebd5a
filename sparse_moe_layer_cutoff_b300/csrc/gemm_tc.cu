// Tensor-core engine of the layer: one persistent, warp-specialised tcgen05 GEMM kernel
// serves every contraction ("Stable LatentMoE": router, down_proj, GroupedExperts gate/up +
// SiTU-GLU, expert down, shared experts, up_proj + shared down), and the dense first-layer
// FFN.  Operands are bf16 (kind::f16), e4m3 for the fp8 routed experts (kind::f8f6f4), or
// MXFP4 weights against e4m3 tokens for the MXFP4 routed experts (kind::mxf8f6f4 with block
// scaling: the weights' ue8m0 block scales go to TMEM by tcgen05.cp before each stage's MMAs).
//
// Weight-stationary tiles.  A tile is 256 weight rows (two MMA operands A0, A1 of M = 128
// rows each) against up to 256 tokens (192 for MXFP4; the MMA's N side, shared by both MMAs), with K
// stepped one 128-byte swizzle row at a time (64 bf16 or 128 e4m3 values):
//   * GLU tiles: A0 = 128 gate rows, A1 = the 128 up rows of the same output features, so
//     one TMEM lane holds both branches of a feature and the SiTU-GLU epilogue needs no
//     exchange between warps;
//   * store tiles: A0, A1 = two consecutive blocks of 128 output rows (A1 is skipped when
//     it lies past the last output row);
//   * an expert segment is covered by full token tiles and one last tile rounded up
//     to a multiple of 16 tokens, so each weight tile is streamed from HBM once per token
//     tile (once per expert at prefill sizes), and each token row is re-read from L2 once
//     per 128 output features.
// Accumulators: TMEM holds 512 fp32 columns in two 256-column slots.  A tile of at most
// 128 tokens takes one slot (A0 in its first 128 columns, A1 in the second), so two such
// tiles double-buffer; a wider tile takes both slots (A0 in slot 0, A1 in slot 1).
// Roles (512 threads): warp 0 streams weight tiles through a 4-stage ring, warp 2 streams
// token tiles through a 3-stage ring (TMA, mbarrier completion), warp 1 owns TMEM and
// issues tcgen05.mma (one thread), warps 4-15 drain the accumulators with tcgen05.ld (three
// warps per TMEM lane quadrant, taking every third 32-token chunk) and write the outputs.
// While a wide tile drains, the next one cannot start, so the epilogue packs its results
// into registers and releases TMEM before the global stores, and SiTU-GLU uses the
// hardware tanh approximation (relative error about 2^-11, below the bf16 rounding of its
// output).  The MXFP4 kernels copy the expert tile schedule into shared memory once per CTA;
// the others read it through L1 (their 256-token stages leave no room).  Every
// mbarrier wait is bounded: on expiry the kernel records the timeout status, drains what it
// issued and returns.
#include <cuda.h>
#include <cuda_fp8.h>

#include <cstring>
#include <new>

#include "common.cuh"
#include "gemm_tc.h"

namespace lmoe {
namespace {

constexpr int kBK = 64;
constexpr int kHalf = 128;                       // weight rows per MMA (M)
constexpr int kTokMax = kTileM;                  // tokens per tile of the grouped MXFP4 GEMMs (MMA N)
constexpr int kTokGroup = kTileWide;             // tokens per tile of the grouped bf16 / e4m3 GEMMs
constexpr int kTokBox = 16;                      // token rows per TMA box
constexpr int kHalfBytes = kHalf * kBK * 2;      // 16 KB
constexpr int kWStageBytes = 2 * kHalfBytes;     // 32 KB of weights per stage
constexpr int kTStagesDefault = 3;
constexpr int kSlotCols = 256;
constexpr int kEpiWarps = 12;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 128 + kEpiThreads;
constexpr int kStaged = 2;                       // 32-token chunks an epilogue warp keeps in registers
constexpr int kSchedMax = 1024;                  // schedule entries kept in shared memory
constexpr int kDenseGroup = 8;                   // token tiles per raster group (dense GEMMs)
constexpr int kPartRows = 2 * kHalf;            // split-K partials: weight rows per tile
constexpr int kPartItem = kPartRows * 256;       // fp32 values per work item ([token][row], <= 256 tokens)
constexpr int kSplitMinKb = 4;                   // k-blocks per split at least
static_assert(kPartItem == kTcPartPerSm, "one work item of partials per SM at most");
constexpr int kMxSfBytes = 512;                  // MXFP4: block scales of 128 rows x 128 K values
// MXFP4 TMEM map: tiles of more than kMxNarrow tokens take both accumulator slots, so columns
// [192, 256) and [448, 512) are never accumulators (tiles hold at most 192 tokens); the weight
// stages' scales use 8 columns each from column 192, the tokens' unit scales 8 from 448.
constexpr int kMxNarrow = 64;
constexpr uint32_t kMxSfaCol = 192;
constexpr uint32_t kMxSfbCol = 448;
// MXFP4 at small batches (no expert with more than kSwapTok tokens): the operands swap roles.  At a
// few tokens an MMA takes the time its A operand needs to leave shared memory (128 rows x 32 bytes
// per K step), and a padded MXFP4 weight tile carries only 2 KB of codes in those 4 KB, so with the
// weights as A the codes would stream at half the bf16 rate.  Here the tokens are A (M = 128 rows;
// rows past the tile's tokens hold stale bytes whose results are never read) and the 256 weight
// rows of a stage are B (N = 256, fetched twice as fast per row).  The accumulator is one
// 256-column slot (lane = token, column = weight row); the tokens' unit scales and the weight
// stages' scales take the columns after it.
constexpr int kSwapTok = 128;
constexpr int kSwapWStages = 5;
constexpr uint32_t kSwapSfaCol = 256;
constexpr uint32_t kSwapSfbCol = 264;

constexpr unsigned long long kTimeoutNs = 2000000000ull;   // 2 s per wait
constexpr unsigned long long kInjectTimeoutNs = 20000000ull; // 20 ms when a timeout is injected

// Shared-memory layout of the grouped (routed experts) and dense launches.  Dense GEMMs and the
// grouped bf16 / e4m3 GEMMs take token tiles of up to 256 (a weight tile's MMAs take about the
// same time for any token count up to 256, so fewer, wider tiles mean less MMA time per token);
// the grouped ones then read their expert schedule through L1.  The grouped MXFP4 GEMMs keep tiles
// of kTokMax tokens (TMEM columns past them hold the block scales) and the schedule in shared
// memory.
// MXV: 0 = bf16 / e4m3 weights, 1 = MXFP4 weights, 2 = MXFP4 weights at small batches with the
// operands swapped (token tiles of at most kSwapTok tokens, held as 128-row MMA operands).
template <bool DENSE, int MXV = 0>
struct Geo {
  static constexpr bool kMx = MXV != 0, kSwap = MXV == 2;
  static constexpr int kTok = DENSE ? 256 : kSwap ? kSwapTok : kMx ? kTokMax : kTokGroup;   // tokens per tile at most
  static constexpr int kWStages = kSwap ? kSwapWStages : 4;      // weight ring (32 KB stages)
  static constexpr int kTStages = kTStagesDefault;               // token ring
  static constexpr bool kSchedSmem = !DENSE && kMx;              // expert schedule in shared memory
  // barriers: W full/empty, T full/empty, TMEM full/empty per slot, drain
  static constexpr int kNumBars = 2 * kWStages + 2 * kTStages + 4 + 1;
  static constexpr int kTStageBytes = kTok * kBK * 2;            // token rows per stage
  static constexpr int kChunks = (kTok / 32 + 2) / 3;           // 32-token chunks per epilogue warp
  static constexpr int kOffT = kWStages * kWStageBytes;
  // MXFP4: the weight stages' block scales (512 bytes per operand) and the tokens' unit scales
  static constexpr int kOffSf = kOffT + kTStages * kTStageBytes;
  static constexpr int kOffSfUnit = kOffSf + (kMx ? kWStages * 2 * kMxSfBytes : 0);
  static constexpr int kOffSched = kOffSfUnit + (kMx ? kMxSfBytes : 0);
  static constexpr int kOffBars = kOffSched + (kSchedSmem ? 2 * kSchedMax * 4 : 0);
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = 1024 + kOffMisc + 16;
  static_assert(kTok % 16 == 0 && kTok <= 256, "MMA N limit");
  static_assert(kChunks <= kStaged + 1, "at most one chunk per warp is written before TMEM is released");
  static_assert(kSmemBytes <= 232448, "shared memory per block");
};

struct TcMaps {
  CUtensorMap w[kMaxKSeg];  // weight (MMA A) maps, one per K segment; GLU: w[0] = gate
  CUtensorMap wup;          // GLU up-branch weights
  CUtensorMap tok;          // token (MMA B) rows, 16-row boxes
};

struct TcParams {
  int nseg;
  int seg_k0[kMaxKSeg + 1];
  int seg_row0[kMaxKSeg];
  int w_group_rows;         // weight rows per group (routed experts), 0 for dense
  int n_feat;               // output features
  int n_fb;                 // feature blocks (256 output rows, or 128 GLU outputs)
  int kblocks;              // K / 64
  int bt;                   // dense: tokens
  int tok_tile;             // tokens per tile: dense (multiple of 16, <= 256), grouped (the schedule's tile size)
  int ksplit;               // dense: work items per tile, each over its own K range (1 = whole K)
  float* part;              // split-K: fp32 accumulators, kPartItem per work item
  const int32_t* seg_off;   // grouped: [G + 1] token segments
  const int32_t* mtile_off; // grouped: [G + 1] prefix of tok_tile-token tiles
  int G;                    // grouped: number of groups, 0 for dense
  void* out;
  long long ldo;
  float* out_t;
  long long ldt;
  const float* bias;
  float beta, beta_u;
  float inv_beta, inv_beta_u;
  // fp8 (e4m3) routed experts: acc * wscale[row] * tscale[perm[slot]] is the gate / up value (GLU,
  // up rows scaled by wscale_up), h is stored as e4m3(act * h_mul); the store kind writes
  // acc * wscale[row] * out_mul
  const float* wscale;
  const float* wscale_up;
  const float* tscale;      // per token (fp8 experts)
  const int32_t* perm;      // routed experts: slot -> token (token scales of the fp8 experts)
  const uint8_t* sf0;       // MXFP4: tiled block scales of the weights (GLU: gate)
  const uint8_t* sf1;       // MXFP4, GLU: up
  float h_mul, out_mul;
  unsigned long long timeout_ns;  // limit of every mbarrier wait
  int inject;               // test hook: the token producer leaves its stages unfilled
  uint32_t* status;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait.  Gives up when the deadline passes (setting abort + timeout status) or,
// if honour_abort, as soon as another role has aborted.  The phase test is inlined and only a
// wait that does not pass at once calls the polling loop: the MMA issuer's loop runs one such
// test per ring stage, and a call there (stack frame and all) slowed the expert GEMMs by 6 %.
__device__ __noinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            uint32_t* status, unsigned long long limit_ns, bool honour_abort) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (global_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t* status,
                                          unsigned long long limit_ns, bool honour_abort = true) {
  return mbar_test(bar, parity) || mbar_wait_poll(bar, parity, abort_flag, status, limit_ns, honour_abort);
}

// 2-D TMA tile load into shared memory, completing on an mbarrier, with an L2 policy.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// 1-D bulk copy global -> shared memory (16-byte aligned, size a multiple of 16), completing on an
// mbarrier, with an L2 policy.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// L2 policies: weights are streamed once (evict first); token rows are re-read by every
// feature block of their tile (evict last).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns of TMEM (this warp's lane quadrant); the caller
// waits with tmem_wait_ld() before reading the registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// kind::f8f6f4 (both operands e4m3, fp32 accumulator): 32 K-elements (32 bytes) per call.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// kind::mxf8f6f4 with block scaling: A = e2m1 weights (each 16-byte shared-memory chunk holds 16
// values in its low 8 bytes), B = e4m3 tokens, 32 K-values per call; A's and B's scales are read
// from TMEM at sfa / sfb, byte sf_id (set in idesc) of each 32-bit word.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc,
                                          uint32_t sfa, uint32_t sfb) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
// 32 rows x 16 bytes of shared memory into 4 TMEM columns, the same 32 rows in each lane quadrant
// (row l to lane l of every quadrant, its 4 words to the 4 columns).
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
template <bool F8>
__device__ __forceinline__ void tc_mma_k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (F8) tc_mma_f8(d, a, b, idesc, acc);
  else tc_mma(d, a, b, idesc, acc);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes
// in 8-row (1024-byte) groups; start address advanced by 32 bytes per K step of 16.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Shared-memory descriptor of a 32-row x 16-byte scale block: no swizzle, 8-row groups 128 bytes
// apart (one 16-byte column, so no leading-dimension offset).
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor: fp32 accumulator, A and B K-major; A / B format 1 = bf16 under
// kind::f16, 0 = e4m3 under kind::f8f6f4.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_e4m3(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// Block-scaled descriptor (kind::mxf8f6f4): A format 5 = e2m1, B format 0 = e4m3, both K-major,
// scale type ue8m0 (bit 23); the scale-factor ids of B (bits 4-5) and A (bits 29-30) are ORed in
// per K step by mx_sf_id.
__device__ __forceinline__ uint32_t idesc_mx(int m, int n) {
  return (5u << 7) | ((uint32_t)(n >> 3) << 17) | (1u << 23) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ uint32_t mx_sf_id(uint32_t j) { return (j << 4) | (j << 29); }
// The same with the operands swapped: A format 0 = e4m3 tokens, B format 5 = e2m1 weights.
__device__ __forceinline__ uint32_t idesc_mx_swap(int m, int n) {
  return (5u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) | ((uint32_t)(m >> 4) << 24);
}

// tanh by the MUFU hardware approximation (PTX tanh.approx.f32).
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// SiTU-GLU from three hardware tanh: g' = beta tanh(g / beta), u' = beta_u tanh(u / beta_u),
// act = g' sigmoid(g') u' with sigmoid(v) = (1 + tanh(v / 2)) / 2.
template <typename P>
__device__ __forceinline__ float situ_glu_fast(float g, float u, const P& p) {
  const float gp = p.beta * tanh_hw(g * p.inv_beta);
  const float up = p.beta_u * tanh_hw(u * p.inv_beta_u);
  const float sg = fmaf(0.5f, tanh_hw(0.5f * gp), 0.5f);
  return gp * sg * up;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// fp32 -> e4m3 (nearest, ties to even, saturating at +-448).
__device__ __forceinline__ uint8_t e4m3_byte(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Barrier over the epilogue warps that also ORs a flag across them.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool flag) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred q, r;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred r, %2, %3, q;\n\tselp.u32 %0, 1, 0, r;\n}"
      : "=r"(res)
      : "r"((uint32_t)flag), "r"(id), "r"(n)
      : "memory");
  return res != 0;
}

// ------------------------------------------------------------------ tile schedule
struct Tile {
  int g, fb, tok0, ntok;
};

__device__ __forceinline__ int num_tiles(const TcParams& p) {
  if (p.G > 0) return p.mtile_off[p.G] * p.n_fb;
  return ((p.bt + p.tok_tile - 1) / p.tok_tile) * p.n_fb;
}

// Grouped: tiles ordered (expert, feature block, token tile), so the CTAs working at the
// same time share weight tiles and token rows in L2; seg/mt are the expert segment and
// tile prefixes (shared memory when they fit).  Dense: token tiles in groups of
// kDenseGroup, feature blocks inside a group.
__device__ __forceinline__ Tile decode_tile(const TcParams& p, const int32_t* seg, const int32_t* mt, int t) {
  Tile r;
  if (p.G > 0) {
    const int q = t / p.n_fb;
    int lo = 0, hi = p.G;                        // largest g with mt[g] <= q
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (mt[mid] <= q) lo = mid; else hi = mid;
    }
    const int m0 = mt[lo];
    const int nt = mt[lo + 1] - m0;
    const int local = t - m0 * p.n_fb;
    r.g = lo;
    r.fb = local / nt;
    const int tb = local - r.fb * nt;
    r.tok0 = seg[lo] + tb * p.tok_tile;
    r.ntok = min(p.tok_tile, seg[lo + 1] - r.tok0);
  } else {
    const int nt = (p.bt + p.tok_tile - 1) / p.tok_tile;
    const int grp = t / (kDenseGroup * p.n_fb);
    const int in = t - grp * kDenseGroup * p.n_fb;
    const int gcnt = min(kDenseGroup, nt - grp * kDenseGroup);
    r.g = 0;
    r.fb = in / gcnt;
    const int tb = grp * kDenseGroup + (in - r.fb * gcnt);
    r.tok0 = tb * p.tok_tile;
    r.ntok = min(p.tok_tile, p.bt - r.tok0);
  }
  return r;
}

// K order of a tile: the feature blocks of one token tile run on neighbouring CTAs at the
// same time and read the same token rows, so each starts its K loop at a different
// offset (evenly spread); every token k-block is then fetched from DRAM by one CTA and
// found in L2 by the others.  The order is fixed per tile, so results are deterministic.
// k_start is computed once per tile; k_at maps the tile's kb-th k-block.
__device__ __forceinline__ int k_start(const TcParams& p, const Tile& tl) {
  return (int)(((long long)tl.fb * p.kblocks) / p.n_fb);
}
__device__ __forceinline__ int k_at(const TcParams& p, int rot, int kb) {
  const int k = kb + rot;
  return k >= p.kblocks ? k - p.kblocks : k;
}

// Work item t of a launch: its tile and k-block range [kb0, kb1).  Split-K launches (dense
// GEMMs with too few tiles to fill the GPU) give each tile ksplit consecutive items, item ks
// covering k-blocks [ks * kblocks / ksplit, (ks + 1) * kblocks / ksplit) in order.
template <bool SPLIT>
__device__ __forceinline__ Tile decode_work(const TcParams& p, const int32_t* seg, const int32_t* mt, int t, int& kb0,
                                            int& kb1) {
  if (!SPLIT) {
    kb0 = 0;
    kb1 = p.kblocks;
    return decode_tile(p, seg, mt, t);
  }
  const int tile = t / p.ksplit, ks = t - tile * p.ksplit;
  kb0 = (int)((long long)ks * p.kblocks / p.ksplit);
  kb1 = (int)((long long)(ks + 1) * p.kblocks / p.ksplit);
  return decode_tile(p, seg, mt, tile);
}

// Weight operands of a tile: GLU always two (gate, up); store / router one or two blocks
// of 128 output rows.
template <int EPI>
__device__ __forceinline__ int tile_halves(const TcParams& p, const Tile& tl) {
  if (EPI == kEpiGlu) return 2;
  return (p.n_feat - tl.fb * 2 * kHalf > kHalf) ? 2 : 1;
}

// TMEM columns of the two accumulators of a tile: narrow tiles (<= 128 tokens) use slot s,
// wide ones both slots.
__device__ __forceinline__ uint32_t acc_col(bool wide, int slot, int h) {
  return wide ? (uint32_t)(h * kSlotCols) : (uint32_t)(slot * kSlotCols + h * kHalf);
}

// ------------------------------------------------------------------ the kernel
template <int EPI, bool F8, bool DENSE, bool SPLIT, int MXV>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  constexpr bool MX = MXV != 0, SWAP = MXV == 2;
  static_assert(!SPLIT || (DENSE && !F8), "split-K covers the dense bf16 GEMMs");
  static_assert(!MX || (F8 && !DENSE && !SPLIT && EPI != kEpiRouter), "MXFP4 covers the routed-expert GEMMs");
  static_assert(kTokMax <= (int)kMxSfaCol, "MXFP4 scale columns lie past the widest accumulator");
  using G = Geo<DENSE, MXV>;
  constexpr int kBKe = F8 ? 2 * kBK : kBK;   // K elements per stage (128-byte rows)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t wbase = base;
  const uint32_t tbase = base + G::kOffT;
  const uint32_t sfbase = base + G::kOffSf;        // MXFP4: block scales of each weight stage
  const uint32_t sfunit = base + G::kOffSfUnit;    // MXFP4: the tokens' unit scales
  int32_t* s_seg = reinterpret_cast<int32_t*>(sbase + G::kOffSched);
  int32_t* s_mt = s_seg + kSchedMax;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + G::kOffBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + G::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
  auto wempty_bar = [&](int s) { return bar0 + 8u * (G::kWStages + s); };
  auto tfull_bar = [&](int s) { return bar0 + 8u * (2 * G::kWStages + s); };
  auto tempty_bar = [&](int s) { return bar0 + 8u * (2 * G::kWStages + G::kTStages + s); };
  auto afull_bar = [&](int a) { return bar0 + 8u * (2 * G::kWStages + 2 * G::kTStages + a); };
  auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * G::kWStages + 2 * G::kTStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * G::kWStages + 2 * G::kTStages + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kWStages; ++s) { mbar_init(wfull_bar(s), 1); mbar_init(wempty_bar(s), 1); }
    for (int s = 0; s < G::kTStages; ++s) { mbar_init(tfull_bar(s), 1); mbar_init(tempty_bar(s), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(afull_bar(a), 1); mbar_init(aempty_bar(a), kEpiWarps); }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const bool sched_smem = G::kSchedSmem && p.G > 0 && p.G < kSchedMax;
  if (sched_smem) {
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
      s_seg[i] = p.seg_off[i];
      s_mt[i] = p.mtile_off[i];
    }
  }
  if (MX) {
    // the token operand carries its per-token scale in the epilogue: its MMA scales are all 2^0
    uint32_t* unit = reinterpret_cast<uint32_t*>(sbase + G::kOffSfUnit);
    for (int i = threadIdx.x; i < kMxSfBytes / 4; i += blockDim.x) unit[i] = 0x7F7F7F7Fu;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(2 * kSlotCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t* seg = sched_smem ? s_seg : p.seg_off;
  const int32_t* mt = sched_smem ? s_mt : p.mtile_off;
  const int nwork = SPLIT ? num_tiles(p) * p.ksplit : num_tiles(p);

  if (warp == 0) {
    // ---------------------------------------------------------------- weight producer
    // Weight operand h of k-block kb of a tile: tensor map and coordinates.
    auto w_src = [&](const Tile& tl, int kb, int h, const CUtensorMap*& m, int& x, int& y) {
      const int k = kb * kBKe;
      if (EPI == kEpiGlu) {
        m = h ? &maps.wup : &maps.w[0];
        x = k;
        y = tl.g * p.w_group_rows + tl.fb * kHalf;
      } else {
        int s = 0;
#pragma unroll
        for (int i = 1; i < kMaxKSeg; ++i)
          if (i < p.nseg && k >= p.seg_k0[i]) s = i;
        m = &maps.w[s];
        x = k - p.seg_k0[s];
        y = p.seg_row0[s] + tl.g * p.w_group_rows + tl.fb * 2 * kHalf + h * kHalf;
      }
    };
    if (lane == 0) {
      const uint64_t wpol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0, pending = 0, pend_parity = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < nwork && !stop; t += gridDim.x) {
        int kb0, kb1;
        const Tile tl = decode_work<SPLIT>(p, seg, mt, t, kb0, kb1);
        const int nh = tile_halves<EPI>(p, tl);
        const int rot = SPLIT ? 0 : k_start(p, tl);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(wempty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { stop = true; break; }
          pending &= ~(1u << stage);
          // MXFP4 boxes write their 8 KB of packed codes into the low halves of 16 KB of chunks
          mbar_expect_tx(wfull_bar(stage), (uint32_t)(nh * (MX ? kHalfBytes / 2 + kMxSfBytes : kHalfBytes)));
          const uint32_t dst = wbase + stage * kWStageBytes;
          const int kq = k_at(p, rot, kb);
          for (int h = 0; h < nh; ++h) {
            const CUtensorMap* m;
            int x, y;
            w_src(tl, kq, h, m, x, y);
            tma_load_2d(dst + h * kHalfBytes, m, x, y, wfull_bar(stage), wpol);
            if (MX) {
              // the 512 scale bytes of these 128 weight rows x 128 K values
              const uint8_t* sf = (EPI == kEpiGlu && h) ? p.sf1 : p.sf0;
              bulk_load(sfbase + (uint32_t)(stage * 2 + h) * kMxSfBytes,
                        sf + ((long long)(y >> 7) * p.kblocks + kq) * kMxSfBytes, kMxSfBytes, wfull_bar(stage), wpol);
            }
          }
          pending |= 1u << stage;
          pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == G::kWStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (stop) {
        // no copy may still be landing in shared memory when the block exits
        for (int s = 0; s < G::kWStages; ++s)
          if (pending & (1u << s)) mbar_wait(wfull_bar(s), (pend_parity >> s) & 1u, abort_flag, p.status, p.timeout_ns, false);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---------------------------------------------------------------- token producer
    const uint64_t tpol = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, pending = 0, pend_parity = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < nwork && !stop; t += gridDim.x) {
      int kb0, kb1;
      const Tile tl = decode_work<SPLIT>(p, seg, mt, t, kb0, kb1);
      const int ntr = (tl.ntok + 15) & ~15;
      const int nbox = ntr / kTokBox;
      const int rot = SPLIT ? 0 : k_start(p, tl);
      if (tl.ntok > G::kTok) {
        // the schedule's tiles never exceed the stages (the host matches them; the swapped MXFP4
        // kernels run only for calls of at most kSwapTok tokens)
        if (lane == 0) {
          atomicOr(p.status, kStatusAssert);
          *abort_flag = 1;
        }
        stop = true;
        break;
      }
      for (int kb = kb0; kb < kb1; ++kb) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(tempty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { stop = true; break; }
        pending &= ~(1u << stage);
        if (p.inject) {
          // test hook: nothing fills this stage, so its consumer's bounded wait runs out
          if (++stage == G::kTStages) { stage = 0; phase ^= 1u; }
          continue;
        }
        if (lane == 0) mbar_expect_tx(tfull_bar(stage), (uint32_t)ntr * (kBK * 2));
        __syncwarp();
        const uint32_t dst = tbase + stage * G::kTStageBytes;
        if (lane < nbox)
          tma_load_2d(dst + lane * (kTokBox * kBK * 2), &maps.tok, k_at(p, rot, kb) * kBKe,
                      tl.tok0 + lane * kTokBox,
                      tfull_bar(stage), tpol);
        pending |= 1u << stage;
        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == G::kTStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (stop && lane == 0) {
      for (int s = 0; s < G::kTStages; ++s)
        if (pending & (1u << s)) mbar_wait(tfull_bar(s), (pend_parity >> s) & 1u, abort_flag, p.status, p.timeout_ns, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int ws = 0, ts = 0, slot = 0;
      uint32_t wph = 0, tph = 0;
      uint32_t aph[2] = {0u, 0u};
      bool stop = false, issued = false;
      if (SWAP) {
        // unit scales of the token operand (A, 128 rows): 4 columns
        tc_cp_sf(tmem_base + kSwapSfaCol, sf_desc(sfunit));
        issued = true;
      } else if (MX) {
        // unit scales of the token operand, 8 columns (up to 256 tokens)
        tc_cp_sf(tmem_base + kMxSfbCol, sf_desc(sfunit));
        tc_cp_sf(tmem_base + kMxSfbCol + 4u, sf_desc(sfunit));
        issued = true;
      }
      for (int t = blockIdx.x; t < nwork && !stop; t += gridDim.x) {
        int kb0, kb1;
        const Tile tl = decode_work<SPLIT>(p, seg, mt, t, kb0, kb1);
        const int ntr = (tl.ntok + 15) & ~15;
        const bool wide = ntr > (MX ? kMxNarrow : kHalf);
        const int nh = tile_halves<EPI>(p, tl);
        if (SWAP) {
          // D[token, weight row] in one 256-column slot: A = the 128-row token stage, B = the
          // stage's nh * 128 weight rows, B's scales moved to this stage's TMEM columns first
          if (!mbar_wait(aempty_bar(0), aph[0] ^ 1u, abort_flag, p.status, p.timeout_ns)) { stop = true; break; }
          tc_fence_after();
          const uint32_t idesc_s = idesc_mx_swap(kHalf, nh * kHalf);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(wfull_bar(ws), wph, abort_flag, p.status, p.timeout_ns) ||
                !mbar_wait(tfull_bar(ts), tph, abort_flag, p.status, p.timeout_ns)) { stop = true; break; }
            tc_fence_after();
            const uint64_t td = smem_desc(tbase + ts * G::kTStageBytes);
            const uint64_t wd = smem_desc(wbase + ws * kWStageBytes);
            const uint32_t sfb = tmem_base + kSwapSfbCol + 8u * ws;
            tc_cp_sf(sfb, sf_desc(sfbase + (uint32_t)(ws * 2) * kMxSfBytes));
            if (nh == 2) tc_cp_sf(sfb + 4u, sf_desc(sfbase + (uint32_t)(ws * 2 + 1) * kMxSfBytes));
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j)
              tc_mma_mx(tmem_base, td + 2u * j, wd + 2u * j, idesc_s | mx_sf_id(j), (kb != kb0 || j != 0) ? 1u : 0u,
                        tmem_base + kSwapSfaCol, sfb);
            issued = true;
            tc_commit(wempty_bar(ws));
            tc_commit(tempty_bar(ts));
            if (++ws == G::kWStages) { ws = 0; wph ^= 1u; }
            if (++ts == G::kTStages) { ts = 0; tph ^= 1u; }
          }
          if (stop) break;
          tc_commit(afull_bar(0));
          aph[0] ^= 1u;
          continue;
        }
        const uint32_t idesc = MX ? idesc_mx(kHalf, ntr) : F8 ? idesc_e4m3(kHalf, ntr) : idesc_bf16(kHalf, ntr);
        if (wide) {
          if (!mbar_wait(aempty_bar(0), aph[0] ^ 1u, abort_flag, p.status, p.timeout_ns) ||
              !mbar_wait(aempty_bar(1), aph[1] ^ 1u, abort_flag, p.status, p.timeout_ns)) { stop = true; break; }
        } else {
          if (!mbar_wait(aempty_bar(slot), aph[slot] ^ 1u, abort_flag, p.status, p.timeout_ns)) { stop = true; break; }
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + acc_col(wide, slot, 0);
        const uint32_t d1 = tmem_base + acc_col(wide, slot, 1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(wfull_bar(ws), wph, abort_flag, p.status, p.timeout_ns) ||
              !mbar_wait(tfull_bar(ts), tph, abort_flag, p.status, p.timeout_ns)) { stop = true; break; }
          tc_fence_after();
          const uint64_t ad = smem_desc(wbase + ws * kWStageBytes);
          const uint64_t bd = smem_desc(tbase + ts * G::kTStageBytes);
          if (MX) {
            // this stage's weight scales into its TMEM columns (issued before, so ordered before,
            // the MMAs that read them; the columns' previous MMAs completed before the stage refilled)
            const uint32_t sfa = tmem_base + kMxSfaCol + 8u * ws;
            tc_cp_sf(sfa, sf_desc(sfbase + (uint32_t)(ws * 2) * kMxSfBytes));
            if (nh == 2) tc_cp_sf(sfa + 4u, sf_desc(sfbase + (uint32_t)(ws * 2 + 1) * kMxSfBytes));
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j)
              tc_mma_mx(d0, ad + 2u * j, bd + 2u * j, idesc | mx_sf_id(j), (kb != kb0 || j != 0) ? 1u : 0u, sfa,
                        tmem_base + kMxSfbCol);
            if (nh == 2) {
              const uint64_t ad1 = ad + (uint64_t)(kHalfBytes >> 4);
#pragma unroll
              for (int j = 0; j < kBK / 16; ++j)
                tc_mma_mx(d1, ad1 + 2u * j, bd + 2u * j, idesc | mx_sf_id(j), (kb != kb0 || j != 0) ? 1u : 0u, sfa + 4u,
                          tmem_base + kMxSfbCol);
            }
          } else {
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j)
              tc_mma_k<F8>(d0, ad + 2u * j, bd + 2u * j, idesc, (kb != kb0 || j != 0) ? 1u : 0u);
            if (nh == 2) {
              const uint64_t ad1 = ad + (uint64_t)(kHalfBytes >> 4);
#pragma unroll
              for (int j = 0; j < kBK / 16; ++j)
                tc_mma_k<F8>(d1, ad1 + 2u * j, bd + 2u * j, idesc, (kb != kb0 || j != 0) ? 1u : 0u);
            }
          }
          issued = true;
          tc_commit(wempty_bar(ws));
          tc_commit(tempty_bar(ts));
          if (++ws == G::kWStages) { ws = 0; wph ^= 1u; }
          if (++ts == G::kTStages) { ts = 0; tph ^= 1u; }
        }
        if (stop) break;
        if (wide) {
          tc_commit(afull_bar(0));
          tc_commit(afull_bar(1));
          aph[0] ^= 1u;
          aph[1] ^= 1u;
        } else {
          tc_commit(afull_bar(slot));
          aph[slot] ^= 1u;
          slot ^= 1;
        }
      }
      if (stop && issued) {
        tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, abort_flag, p.status, p.timeout_ns, false);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int sub = (warp - 4) >> 2;        // which 32-token chunks: sub, sub + 3, ...
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    int slot = 0;
    uint32_t aph[2] = {0u, 0u};
    for (int t = blockIdx.x; t < nwork; t += gridDim.x) {
      int kb0, kb1;
      const Tile tl = decode_work<SPLIT>(p, seg, mt, t, kb0, kb1);
      const int ntr = (tl.ntok + 15) & ~15;
      const bool wide = ntr > (MX ? kMxNarrow : kHalf);
      const int nh = tile_halves<EPI>(p, tl);
      if (SWAP) {
        // lane = token q * 32 + lane of the tile; this warp takes the 32-column chunks sub, sub + 3, ...
        // GLU: gate columns [0, 128), up columns [128, 256) -> 32 e4m3 activations per chunk;
        // store: nh * 128 output columns -> 32 bf16 values per chunk.  TMEM is released before the
        // stores; each lane then writes its token's row segments (32 or 64 contiguous bytes).
        const bool ok = mbar_wait(afull_bar(0), aph[0], abort_flag, p.status, p.timeout_ns);
        if (named_sync_or(1, kEpiThreads, !ok || *abort_flag)) break;
        tc_fence_after();
        const int tok = q * 32 + lane;
        const bool live = tok < tl.ntok;
        uint32_t res[3][16];
        const int nchunk = EPI == kEpiGlu ? 4 : nh * 4;
        if (EPI == kEpiGlu) {
          const float ts = live ? p.tscale[p.perm[tl.tok0 + tok]] : 0.f;
#pragma unroll
          for (int nc = 0; nc < 2; ++nc) {
            const int c = sub + 3 * nc;
            if (c >= nchunk) break;
            uint32_t g[32], u[32];
            tmem_ld32(lane_base + c * 32, g);
            tmem_ld32(lane_base + kHalf + c * 32, u);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              uint32_t word = 0;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const float a = situ_glu_fast(__uint_as_float(g[j + b]) * ts, __uint_as_float(u[j + b]) * ts, p);
                word |= (uint32_t)e4m3_byte(a * p.h_mul) << (8 * b);
              }
              res[nc][j >> 2] = word;
            }
          }
        } else {
#pragma unroll
          for (int nc = 0; nc < 3; ++nc) {
            const int c = sub + 3 * nc;
            if (c >= nchunk) break;
            uint32_t v[32];
            tmem_ld32(lane_base + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              res[nc][j] = pack_bf16x2(__uint_as_float(v[2 * j]) * p.out_mul, __uint_as_float(v[2 * j + 1]) * p.out_mul);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aempty_bar(0));
        aph[0] ^= 1u;
        if (live) {
          const long long row = tl.tok0 + tok;
          if (EPI == kEpiGlu) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int c = sub + 3 * k;
              if (c >= nchunk) break;
              uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + row * p.ldo + tl.fb * kHalf + c * 32);
              o[0] = make_uint4(res[k][0], res[k][1], res[k][2], res[k][3]);
              o[1] = make_uint4(res[k][4], res[k][5], res[k][6], res[k][7]);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 3; ++k) {
              const int c = sub + 3 * k;
              if (c >= nchunk) break;
              uint4* o = reinterpret_cast<uint4*>(static_cast<bf16*>(p.out) + row * p.ldo + tl.fb * 2 * kHalf + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) o[v] = make_uint4(res[k][4 * v], res[k][4 * v + 1], res[k][4 * v + 2], res[k][4 * v + 3]);
            }
          }
        }
        continue;
      }
      bool ok;
      if (wide) ok = mbar_wait(afull_bar(0), aph[0], abort_flag, p.status, p.timeout_ns) &&
                     mbar_wait(afull_bar(1), aph[1], abort_flag, p.status, p.timeout_ns);
      else ok = mbar_wait(afull_bar(slot), aph[slot], abort_flag, p.status, p.timeout_ns);
      if (named_sync_or(1, kEpiThreads, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t c0 = lane_base + acc_col(wide, slot, 0);
      const uint32_t c1 = lane_base + acc_col(wide, slot, 1);
      const int nchunks = (tl.ntok + 31) >> 5;
      const int fbase = EPI == kEpiGlu ? tl.fb * kHalf + q * 32 + lane : tl.fb * 2 * kHalf + q * 32 + lane;
      // Writes one packed 32-token chunk of output half h (bf16 pairs of consecutive tokens,
      // or e4m3 quads for the fp8 GLU) to its rows.
      auto store_chunk = [&](int c, int h, const uint32_t* w) {
        const int nj = min(32, tl.ntok - c * 32);
        const int fout = fbase + h * kHalf;
        if (fout >= p.n_feat) return;
        if (F8 && EPI == kEpiGlu) {
          uint8_t* o = static_cast<uint8_t*>(p.out) + (long long)(tl.tok0 + c * 32) * p.ldo + fout;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nj) o[(long long)j * p.ldo] = (uint8_t)(w[j >> 2] >> (8 * (j & 3)));
        } else {
          bf16* o = static_cast<bf16*>(p.out) + (long long)(tl.tok0 + c * 32) * p.ldo + fout;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nj) o[(long long)j * p.ldo] = __ushort_as_bfloat16((unsigned short)((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu)));
        }
      };
      // Results of this warp's first kStaged chunks stay in registers and are written after
      // TMEM is released; later chunks (tiles of more than 192 tokens) are written at once.
      uint32_t res[kStaged][2][16];
      if (SPLIT) {
        // the raw fp32 accumulators of this work item, part[t][token][row] (row = 128 h + TMEM
        // lane): for each token the 32 lanes of a warp write 128 consecutive bytes
        float* wp = p.part + (long long)t * kPartItem;
        for (int c = sub; c < nchunks; c += 3) {
          const int nj = min(32, tl.ntok - c * 32);
          for (int h = 0; h < nh; ++h) {
            uint32_t v[32];
            tmem_ld32((h ? c1 : c0) + c * 32, v);
            tmem_wait_ld();
            float* o = wp + (long long)(c * 32) * kPartRows + h * kHalf + q * 32 + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nj) o[j * kPartRows] = __uint_as_float(v[j]);
          }
        }
      } else if (EPI == kEpiGlu) {
        // fp8: per-row weight scales of this lane's feature (gate and up rows)
        float sg = 1.f, su = 1.f;
        if (F8 && !MX) {
          const int fo = tl.fb * kHalf + q * 32 + lane;
          if (fo < p.n_feat) {
            sg = p.wscale[(long long)tl.g * p.w_group_rows + fo];
            su = p.wscale_up[(long long)tl.g * p.w_group_rows + fo];
          }
        }
#pragma unroll
        for (int ci = 0; ci < G::kChunks; ++ci) {
          const int c = sub + 3 * ci;
          if (c < nchunks) {
            uint32_t g[32], u[32], w[16];
            tmem_ld32(c0 + c * 32, g);
            tmem_ld32(c1 + c * 32, u);
            float ts = 1.f;   // fp8: this lane's token scale (lane j holds token j of the chunk)
            if (F8 && c * 32 + lane < tl.ntok) ts = p.tscale[p.perm[tl.tok0 + c * 32 + lane]];
            tmem_wait_ld();
            if (F8) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                uint32_t word = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                  const float tj = __shfl_sync(0xffffffffu, ts, j + b);
                  const float a = situ_glu_fast(__uint_as_float(g[j + b]) * (sg * tj),
                                                __uint_as_float(u[j + b]) * (su * tj), p);
                  word |= (uint32_t)e4m3_byte(a * p.h_mul) << (8 * b);
                }
                w[j >> 2] = word;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[j] = pack_bf16x2(situ_glu_fast(__uint_as_float(g[2 * j]), __uint_as_float(u[2 * j]), p),
                                   situ_glu_fast(__uint_as_float(g[2 * j + 1]), __uint_as_float(u[2 * j + 1]), p));
            }
            if (ci < kStaged) {
#pragma unroll
              for (int j = 0; j < 16; ++j) res[ci < kStaged ? ci : 0][0][j] = w[j];
            } else {
              store_chunk(c, 0, w);
            }
          }
        }
      } else if (EPI == kEpiStore) {
#pragma unroll
        for (int ci = 0; ci < G::kChunks; ++ci) {
          const int c = sub + 3 * ci;
          if (c < nchunks) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (h < nh) {
                uint32_t v[32], w[16];
                tmem_ld32((h ? c1 : c0) + c * 32, v);
                float sc = 1.f;   // fp8: row scale times the activation scale
                if (F8) {
                  const int fo = tl.fb * 2 * kHalf + h * kHalf + q * 32 + lane;
                  if (fo < p.n_feat) sc = (MX ? 1.f : p.wscale[(long long)tl.g * p.w_group_rows + fo]) * p.out_mul;
                }
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  w[j] = pack_bf16x2(__uint_as_float(v[2 * j]) * sc, __uint_as_float(v[2 * j + 1]) * sc);
                if (ci < kStaged) {
#pragma unroll
                  for (int j = 0; j < 16; ++j) res[ci < kStaged ? ci : 0][h][j] = w[j];
                } else {
                  store_chunk(c, h, w);
                }
              }
            }
          }
        }
      } else {
        // router: fp32 logits and their transpose, written straight from TMEM
        const int f0 = tl.fb * 2 * kHalf + q * 32 + lane;
        for (int c = sub; c < nchunks; c += 3) {
          const int nj = min(32, tl.ntok - c * 32);
          for (int h = 0; h < nh; ++h) {
            uint32_t v[32];
            tmem_ld32((h ? c1 : c0) + c * 32, v);
            tmem_wait_ld();
            const int fout = f0 + h * kHalf;
            if (fout >= p.n_feat) continue;
            const long long row0 = tl.tok0 + c * 32;
            const float bias = p.bias ? p.bias[fout] : 0.f;
            float* o = static_cast<float*>(p.out) + row0 * p.ldo + fout;
            float* ot = p.out_t + (long long)fout * p.ldt + row0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v[j] = __float_as_uint(__uint_as_float(v[j]) + bias);
              if (j < nj) o[(long long)j * p.ldo] = __uint_as_float(v[j]);
            }
            // the transposed row: this lane's 32 consecutive tokens, 16-byte stores when aligned
            if (nj == 32 && (reinterpret_cast<uintptr_t>(ot) & 15u) == 0) {
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<uint4*>(ot + j) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nj) ot[j] = __uint_as_float(v[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (wide) { mbar_arrive(aempty_bar(0)); mbar_arrive(aempty_bar(1)); }
        else mbar_arrive(aempty_bar(slot));
      }
      if (EPI != kEpiRouter && !SPLIT) {
#pragma unroll
        for (int ci = 0; ci < kStaged; ++ci) {
          const int c = sub + 3 * ci;
          if (c >= nchunks) continue;
#pragma unroll
          for (int h = 0; h < (EPI == kEpiGlu ? 1 : 2); ++h)
            if (h < nh) store_chunk(c, h, res[ci][h]);
        }
      }
      if (wide) { aph[0] ^= 1u; aph[1] ^= 1u; }
      else { aph[slot] ^= 1u; slot ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(2 * kSlotCols));
}

// Split-K reduction and epilogue: sums the ksplit partial accumulators of every (tile, token,
// weight row) in the fixed order ks = 0, 1, ... (so results are deterministic) and applies the
// launch's epilogue: bf16 store, SiTU-GLU of the gate and up sums, or the router's fp32 logits
// plus bias and their transposed copy.  tt = tokens per tile index range (<= tok_tile).
template <int EPI>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const TcParams p, int tt) {
  constexpr int R = EPI == kEpiGlu ? kHalf : 2 * kHalf;   // output rows of a tile
  const long long total = (long long)num_tiles(p) * tt * R;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i % R);
    const long long q = i / R;
    const int tok = (int)(q % tt);
    const int T = (int)(q / tt);
    const Tile tl = decode_tile(p, nullptr, nullptr, T);
    if (tok >= tl.ntok) continue;
    const int f = EPI == kEpiGlu ? tl.fb * kHalf + r : tl.fb * 2 * kHalf + r;
    if (f >= p.n_feat) continue;
    const float* src = p.part + (long long)T * p.ksplit * kPartItem + (long long)tok * kPartRows + r;
    float s0 = 0.f, s1 = 0.f;
    for (int ks = 0; ks < p.ksplit; ++ks) {
      s0 += src[(long long)ks * kPartItem];
      if (EPI == kEpiGlu) s1 += src[(long long)ks * kPartItem + kHalf];
    }
    const long long row = tl.tok0 + tok;
    if (EPI == kEpiGlu) {
      static_cast<bf16*>(p.out)[row * p.ldo + f] = __float2bfloat16_rn(situ_glu_fast(s0, s1, p));
    } else if (EPI == kEpiStore) {
      static_cast<bf16*>(p.out)[row * p.ldo + f] = __float2bfloat16_rn(s0);
    } else {
      const float v = s0 + (p.bias ? p.bias[f] : 0.f);
      static_cast<float*>(p.out)[row * p.ldo + f] = v;
      p.out_t[(long long)f * p.ldt + row] = v;
    }
  }
}

// Routed-expert token rows in slot order: zp[slot] = rows[perm[slot]] (z, or its e4m3 copy);
// one warp per row, 16-byte vectors (HBM-bound: each row is read from L2-resident rows and
// written once).  A lane issues its loads kGatherBatch at a time before storing them, so
// enough bytes are in flight to cover the L2 latency.
constexpr int kGatherBatch = 7;   // 3584-wide rows: 14 (bf16) or 7 (e4m3) vectors per lane
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ rows, const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ offsets, int n_experts,
                                                          int vec_per_row, uint4* __restrict__ zp) {
  const int nslots = offsets[n_experts];
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int slot = blockIdx.x * wpb + (threadIdx.x >> 5); slot < nslots; slot += gridDim.x * wpb) {
    const uint4* src = rows + (long long)perm[slot] * vec_per_row;
    uint4* dst = zp + (long long)slot * vec_per_row;
    int v = lane;
    for (; v + 32 * (kGatherBatch - 1) < vec_per_row; v += 32 * kGatherBatch) {
      uint4 r[kGatherBatch];
#pragma unroll
      for (int i = 0; i < kGatherBatch; ++i) r[i] = src[v + 32 * i];
#pragma unroll
      for (int i = 0; i < kGatherBatch; ++i) dst[v + 32 * i] = r[i];
    }
    for (; v < vec_per_row; v += 32) dst[v] = src[v];
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    cudaGetLastError();
  }
  return fn;
}

// 2-D map over rows x cols (row stride ld elements) of bf16 (box 64 columns) or of bytes
// (e4m3, box 128 columns), box_rows rows, 128-byte swizzle; rows past the end read as zero.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_rows,
              bool u8 = false) {
  EncodeTiledFn enc = encoder();
  if (!enc || rows <= 0) return false;
  const int esz = u8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over rows x cols e2m1 codes packed two per byte (row stride cols / 2 bytes): boxes of
// 128 values (64 bytes) x box_rows rows, each 8-byte group of 16 values landing in the low half of
// a 16-byte shared-memory chunk (16U4_ALIGN16B), 128-byte swizzle: the shared-memory image of a
// box is that of a 128-column box of bytes.
bool make_map_fp4(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn enc = encoder();
  if (!enc || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token tile of a dense GEMM: the multiple of 16 in [128, 256] that minimises
// waves x (tile + a fixed per-tile cost of 32 tokens), so the last wave of the persistent
// grid is nearly full (e.g. the 8192-token router: 172 tiles of 192 tokens leave most of
// the second wave idle; 256 tiles of 128 fill it, and narrow tiles double-buffer TMEM).
int dense_tok_tile(int bt, int n_fb, int grid) {
  constexpr int kMax = Geo<true>::kTok;
  int best = kMax;
  long long best_cost = -1;
  for (int tt = kMax; tt >= 128; tt -= 16) {
    const long long tiles = (long long)((bt + tt - 1) / tt) * n_fb;
    const long long waves = (tiles + grid - 1) / grid;
    const long long cost = waves * (tt + 32);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = tt; }
  }
  return best;
}

template <int EPI, bool F8, bool DENSE, bool SPLIT = false, int MXV = 0>
cudaError_t launch_kernel(const TcMaps& maps, const TcParams& p, int grid, cudaStream_t st) {
  tc_gemm_kernel<EPI, F8, DENSE, SPLIT, MXV><<<grid, kThreads, Geo<DENSE, MXV>::kSmemBytes, st>>>(maps, p);
  return cudaGetLastError();
}

// A dense split-K GEMM: the partial products, then their reduction with the epilogue.
template <int EPI>
cudaError_t launch_split(const TcMaps& maps, const TcParams& p, int grid, int sm_count, cudaStream_t st) {
  cudaError_t e = launch_kernel<EPI, false, true, true>(maps, p, grid, st);
  if (e != cudaSuccess) return e;
  const int tt = p.tok_tile < p.bt ? p.tok_tile : p.bt;
  const long long total = (long long)((p.bt + p.tok_tile - 1) / p.tok_tile) * p.n_fb * tt * (EPI == kEpiGlu ? kHalf : 2 * kHalf);
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)sm_count * 8) blocks = (long long)sm_count * 8;
  splitk_reduce_kernel<EPI><<<(int)blocks, 256, 0, st>>>(p, tt);
  return cudaGetLastError();
}

// One GEMM: the persistent kernel with grid = SMs (fewer when a dense GEMM has fewer work
// items).  A dense GEMM with at most half as many tiles as SMs and a partial buffer
// (p.part) is split along K into up to SMs / tiles work items per tile (each of at least
// kSplitMinKb k-blocks) and reduced by a second kernel.  *n = kernels launched.
cudaError_t launch_tc(const TcMaps& maps, TcParams& p, int epi, int sm_count, cudaStream_t st, bool f8, int* n,
                      int mxv = 0) {
  *n = 0;
  p.ksplit = 1;
  if (p.G == 0) p.tok_tile = dense_tok_tile(p.bt, p.n_fb, sm_count);
  int grid = sm_count;
  if (p.G == 0) {
    const long long tiles = (long long)((p.bt + p.tok_tile - 1) / p.tok_tile) * p.n_fb;
    if (p.part && tiles > 0 && 2 * tiles <= sm_count) {
      long long s = sm_count / tiles;
      if (s > p.kblocks / kSplitMinKb) s = p.kblocks / kSplitMinKb;
      if (s >= 2) p.ksplit = (int)s;
    }
    if (tiles * p.ksplit < grid) grid = (int)(tiles * p.ksplit);
  }
  if (grid <= 0) return cudaSuccess;
  *n = p.ksplit > 1 ? 2 : 1;
  if (mxv == 2) {   // the MXFP4 routed experts at small batches, operands swapped (at most kSwapTok tokens per expert)
    if (epi == kEpiGlu) return launch_kernel<kEpiGlu, true, false, false, 2>(maps, p, grid, st);
    return launch_kernel<kEpiStore, true, false, false, 2>(maps, p, grid, st);
  }
  if (mxv == 1) {   // the MXFP4 routed experts (grouped)
    if (epi == kEpiGlu) return launch_kernel<kEpiGlu, true, false, false, 1>(maps, p, grid, st);
    return launch_kernel<kEpiStore, true, false, false, 1>(maps, p, grid, st);
  }
  if (f8) {   // the fp8 routed experts (grouped)
    if (epi == kEpiGlu) return launch_kernel<kEpiGlu, true, false>(maps, p, grid, st);
    return launch_kernel<kEpiStore, true, false>(maps, p, grid, st);
  }
  if (p.G > 0) {
    if (epi == kEpiGlu) return launch_kernel<kEpiGlu, false, false>(maps, p, grid, st);
    return launch_kernel<kEpiStore, false, false>(maps, p, grid, st);
  }
  if (p.ksplit > 1) {
    switch (epi) {
      case kEpiStore: return launch_split<kEpiStore>(maps, p, grid, sm_count, st);
      case kEpiGlu: return launch_split<kEpiGlu>(maps, p, grid, sm_count, st);
      default: return launch_split<kEpiRouter>(maps, p, grid, sm_count, st);
    }
  }
  switch (epi) {
    case kEpiStore: return launch_kernel<kEpiStore, false, true>(maps, p, grid, st);
    case kEpiGlu: return launch_kernel<kEpiGlu, false, true>(maps, p, grid, st);
    default: return launch_kernel<kEpiRouter, false, true>(maps, p, grid, st);
  }
}

template <int EPI, bool F8, bool DENSE, bool SPLIT = false, int MXV = 0>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(tc_gemm_kernel<EPI, F8, DENSE, SPLIT, MXV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Geo<DENSE, MXV>::kSmemBytes);
}

// Raises the dynamic shared-memory limit of every kernel instance a plan launches.
cudaError_t prepare_kernels(bool f8, bool mx = false) {
  cudaError_t e = set_smem<kEpiStore, false, true>();
  if (e == cudaSuccess) e = set_smem<kEpiGlu, false, true>();
  if (e == cudaSuccess) e = set_smem<kEpiRouter, false, true>();
  if (e == cudaSuccess) e = set_smem<kEpiStore, false, true, true>();
  if (e == cudaSuccess) e = set_smem<kEpiGlu, false, true, true>();
  if (e == cudaSuccess) e = set_smem<kEpiRouter, false, true, true>();
  if (e == cudaSuccess) e = set_smem<kEpiStore, false, false>();
  if (e == cudaSuccess) e = set_smem<kEpiGlu, false, false>();
  if (e == cudaSuccess && f8) e = set_smem<kEpiGlu, true, false>();
  if (e == cudaSuccess && f8) e = set_smem<kEpiStore, true, false>();
  if (e == cudaSuccess && mx) e = set_smem<kEpiGlu, true, false, false, 1>();
  if (e == cudaSuccess && mx) e = set_smem<kEpiStore, true, false, false, 1>();
  if (e == cudaSuccess && mx) e = set_smem<kEpiGlu, true, false, false, 2>();
  if (e == cudaSuccess && mx) e = set_smem<kEpiStore, true, false, false, 2>();
  return e;
}

}  // namespace

struct TcPlan {
  lmoe_config cfg;
  int max_bt;
  int sm_count;
  TcBuffers buf;
  bool f8;                                                  // e4m3 token rows and h (fp8 or MXFP4 experts)
  bool mx;                                                  // MXFP4 expert weights
  CUtensorMap m_gate8, m_up8, m_edown8, m_zq8, m_h8;        // their weights, token rows, h
  const float *s_gate, *s_up, *s_down;                      // fp8: per-row weight scales
  const uint8_t *sf_gate, *sf_up, *sf_down;                 // MXFP4: tiled block scales
  float h_mul, h_scale;                                     // fixed activation scale (SiTU-GLU bound)
  bool inject;                                              // test hook armed for the next expert gate/up
  CUtensorMap m_router, m_down, m_gate, m_up, m_edown, m_shg, m_shu, m_wup, m_shd;  // weights
  CUtensorMap m_zp, m_h, m_cat;                                                       // workspace
};

lmoe_status tc_plan_create(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_fp8_experts* f8,
                           const lmoe_mxfp4_experts* mx, int max_bt, int sm_count, const TcBuffers& buf, TcPlan** plan) {
  *plan = nullptr;
  TcPlan* pl = new (std::nothrow) TcPlan();
  if (!pl) return LMOE_ERR_OOM;
  pl->cfg = *cfg;
  pl->max_bt = max_bt;
  pl->sm_count = sm_count;
  pl->buf = buf;
  const lmoe_config& c = *cfg;
  const long long E = c.n_experts, d = c.d, L = c.latent, I = c.expert_inter, S = c.n_shared, Is = c.shared_inter;
  const long long ldc = L + S * Is;
  const long long slots = (long long)max_bt * c.top_k;
  pl->f8 = f8 != nullptr || mx != nullptr;
  pl->mx = mx != nullptr;
  bool ok = make_map(&pl->m_router, w->w_router, E, d, d, kHalf) && make_map(&pl->m_down, w->w_down, L, d, d, kHalf);
  if (pl->f8) {
    if (pl->mx) {
      ok = ok && make_map_fp4(&pl->m_gate8, mx->exp_gate, E * I, L, kHalf) &&
           make_map_fp4(&pl->m_up8, mx->exp_up, E * I, L, kHalf) && make_map_fp4(&pl->m_edown8, mx->exp_down, E * L, I, kHalf);
      pl->sf_gate = static_cast<const uint8_t*>(mx->gate_sf);
      pl->sf_up = static_cast<const uint8_t*>(mx->up_sf);
      pl->sf_down = static_cast<const uint8_t*>(mx->down_sf);
    } else {
      ok = ok && make_map(&pl->m_gate8, f8->exp_gate, E * I, L, L, kHalf, true) &&
           make_map(&pl->m_up8, f8->exp_up, E * I, L, L, kHalf, true) &&
           make_map(&pl->m_edown8, f8->exp_down, E * L, I, I, kHalf, true);
      pl->s_gate = f8->gate_scale;
      pl->s_up = f8->up_scale;
      pl->s_down = f8->down_scale;
    }
    ok = ok && make_map(&pl->m_zq8, buf.zp, slots, L, L, kTokBox, true) && make_map(&pl->m_h8, buf.h, slots, I, I, kTokBox, true);
    const float bound = c.beta * c.beta_u;   // |SiTU-GLU| < beta * beta_u
    pl->h_mul = 448.0f / bound;
    pl->h_scale = bound / 448.0f;
  } else {
    ok = ok && make_map(&pl->m_gate, w->exp_gate, E * I, L, L, kHalf) && make_map(&pl->m_up, w->exp_up, E * I, L, L, kHalf) &&
         make_map(&pl->m_edown, w->exp_down, E * L, I, I, kHalf);
  }
  ok = ok &&
            make_map(&pl->m_shg, w->sh_gate, S * Is, d, d, kHalf) && make_map(&pl->m_shu, w->sh_up, S * Is, d, d, kHalf) &&
            make_map(&pl->m_wup, w->w_up, d, L, L, kHalf) && make_map(&pl->m_shd, w->sh_down, S * d, Is, Is, kHalf) &&
            make_map(&pl->m_zp, buf.zp, slots, L, L, kTokBox) && make_map(&pl->m_h, buf.h, slots, I, I, kTokBox) &&
            make_map(&pl->m_cat, buf.cat, max_bt, ldc, ldc, kTokBox);
  if (!ok) {
    delete pl;
    return LMOE_ERR_CUDA;
  }
  cudaError_t e = prepare_kernels(pl->f8, pl->mx);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete pl;
    return LMOE_ERR_CUDA;
  }
  *plan = pl;
  return LMOE_OK;
}

void tc_plan_destroy(TcPlan* plan) { delete plan; }

void tc_inject_wait_timeout(TcPlan* plan) { plan->inject = true; }

int tc_group_tile(const TcPlan* plan) { return plan->mx ? kTileM : kTileWide; }

cudaError_t tc_gather_tokens(TcPlan* pl, const GemmArgs& a, cudaStream_t st, int* n) {
  const lmoe_config& c = pl->cfg;
  const void* rows = pl->buf.z;
  int vec = c.latent / 8;
  *n = 1;
  if (pl->f8) {
    cudaError_t e = launch_quantize_rows(pl->buf.z, a.bt_tokens, c.latent, pl->buf.zq, pl->buf.tscale,
                                         pl->sm_count * 8, st);
    if (e != cudaSuccess) return e;
    rows = pl->buf.zq;
    vec = c.latent / 16;
    *n = 2;
  }
  gather_rows_kernel<<<pl->sm_count * 8, 256, 0, st>>>(static_cast<const uint4*>(rows), a.a_rows, a.seg_off, a.G, vec,
                                                       static_cast<uint4*>(pl->buf.zp));
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(TcPlan* pl, const GemmArgs& a, cudaStream_t st, int* n) {
  *n = 0;
  const lmoe_config& c = pl->cfg;
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.nseg = 1;
  p.seg_k0[0] = 0;
  p.seg_k0[1] = a.K;
  p.n_feat = a.N;
  p.kblocks = a.K / kBK;
  p.out = a.out;
  p.ldo = a.ldo;
  p.beta = a.beta;
  p.beta_u = a.beta_u;
  p.inv_beta = 1.0f / a.beta;
  p.inv_beta_u = 1.0f / a.beta_u;
  p.status = pl->buf.status;
  p.timeout_ns = kTimeoutNs;
  p.part = pl->buf.part;   // dense GEMMs may split K (launch_tc decides)
  int epi = a.epi;
  bool ok = true, f8 = false;
  switch (a.op) {
    case kOpRouter:
      maps.w[0] = pl->m_router;
      ok = make_map(&maps.tok, a.A, a.M, a.K, a.lda, kTokBox);
      p.bt = a.M;
      p.out_t = a.out_t;
      p.ldt = a.ldt;
      p.bias = a.bias;
      break;
    case kOpDown:
      maps.w[0] = pl->m_down;
      ok = make_map(&maps.tok, a.A, a.M, a.K, a.lda, kTokBox);
      p.bt = a.M;
      break;
    case kOpSharedGateUp:
      maps.w[0] = pl->m_shg;
      maps.wup = pl->m_shu;
      ok = make_map(&maps.tok, a.A, a.M, a.K, a.lda, kTokBox);
      p.bt = a.M;
      break;
    case kOpFinal:
      maps.w[0] = pl->m_wup;
      maps.tok = pl->m_cat;
      p.bt = a.M;
      p.nseg = a.nseg;
      for (int s = 0; s < a.nseg; ++s) {
        if (s > 0) maps.w[s] = pl->m_shd;
        p.seg_k0[s] = a.seg_k0[s];
        p.seg_row0[s] = (int)a.seg_row0[s];
      }
      p.seg_k0[a.nseg] = a.K;
      break;
    case kOpExpertGateUp: {
      if (pl->inject) {
        p.inject = 1;
        p.timeout_ns = kInjectTimeoutNs;
        pl->inject = false;
      }
      // token rows: the slot-ordered copy tc_gather_tokens made (bf16, or e4m3 with per-token scales)
      if (pl->f8) {
        maps.w[0] = pl->m_gate8;
        maps.wup = pl->m_up8;
        maps.tok = pl->m_zq8;
        p.wscale = pl->s_gate;
        p.wscale_up = pl->s_up;
        p.sf0 = pl->sf_gate;
        p.sf1 = pl->sf_up;
        p.tscale = pl->buf.tscale;
        p.perm = a.a_rows;
        p.h_mul = pl->h_mul;
        p.kblocks = a.K / (2 * kBK);
        f8 = true;
      } else {
        maps.w[0] = pl->m_gate;
        maps.wup = pl->m_up;
        maps.tok = pl->m_zp;
      }
      p.w_group_rows = c.expert_inter;
      p.seg_off = a.seg_off;
      p.mtile_off = a.mtile_off;
      p.G = a.G;
      p.tok_tile = tc_group_tile(pl);
      break;
    }
    case kOpExpertDown:
      if (pl->f8) {
        maps.w[0] = pl->m_edown8;
        maps.tok = pl->m_h8;
        p.wscale = pl->s_down;
        p.sf0 = pl->sf_down;
        p.out_mul = pl->h_scale;
        p.kblocks = a.K / (2 * kBK);
        f8 = true;
      } else {
        maps.w[0] = pl->m_edown;
        maps.tok = pl->m_h;
      }
      p.w_group_rows = c.latent;
      p.seg_off = a.seg_off;
      p.mtile_off = a.mtile_off;
      p.G = a.G;
      p.tok_tile = tc_group_tile(pl);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  p.n_fb = epi == kEpiGlu ? (a.N + kHalf - 1) / kHalf : (a.N + 2 * kHalf - 1) / (2 * kHalf);
  // a call of at most kSwapTok tokens gives no expert more (top-K experts are distinct per token)
  return launch_tc(maps, p, epi, pl->sm_count, st, f8, n, !(f8 && pl->mx) ? 0 : a.bt_tokens <= kSwapTok ? 2 : 1);
}

// ------------------------------------------------------------------ dense SiTU-GLU FFN
struct TcFfnPlan {
  int d, inter, sm_count;
  float beta, beta_u;
  void* h;
  uint32_t* status;
  CUtensorMap m_gate, m_up, m_down, m_h;
};

lmoe_status tc_ffn_create(int d, int inter, float beta, float beta_u, const void* w_gate, const void* w_up,
                          const void* w_down, int max_bt, int sm_count, void* h, uint32_t* status, TcFfnPlan** plan) {
  *plan = nullptr;
  TcFfnPlan* pl = new (std::nothrow) TcFfnPlan();
  if (!pl) return LMOE_ERR_OOM;
  pl->d = d;
  pl->inter = inter;
  pl->sm_count = sm_count;
  pl->beta = beta;
  pl->beta_u = beta_u;
  pl->h = h;
  pl->status = status;
  const bool ok = make_map(&pl->m_gate, w_gate, inter, d, d, kHalf) && make_map(&pl->m_up, w_up, inter, d, d, kHalf) &&
                  make_map(&pl->m_down, w_down, d, inter, inter, kHalf) &&
                  make_map(&pl->m_h, h, max_bt, inter, inter, kTokBox);
  cudaError_t e = ok ? prepare_kernels(false) : cudaErrorInvalidValue;
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete pl;
    return LMOE_ERR_CUDA;
  }
  *plan = pl;
  return LMOE_OK;
}

void tc_ffn_destroy(TcFfnPlan* plan) { delete plan; }

// h = act(x W_gate^T, x W_up^T), then out = h W_down^T: two launches of the GEMM kernel.
cudaError_t tc_ffn_forward(TcFfnPlan* pl, const void* x, int bt, void* out, cudaStream_t st) {
  TcMaps maps;
  TcParams p;
  for (int pass = 0; pass < 2; ++pass) {
    memset(&maps, 0, sizeof(maps));
    memset(&p, 0, sizeof(p));
    p.nseg = 1;
    p.bt = bt;
    p.beta = pl->beta;
    p.beta_u = pl->beta_u;
    p.inv_beta = 1.0f / pl->beta;
    p.inv_beta_u = 1.0f / pl->beta_u;
    p.status = pl->status;
    p.timeout_ns = kTimeoutNs;
    if (pass == 0) {
      maps.w[0] = pl->m_gate;
      maps.wup = pl->m_up;
      if (!make_map(&maps.tok, x, bt, pl->d, pl->d, kTokBox)) return cudaErrorInvalidValue;
      p.seg_k0[1] = pl->d;
      p.n_feat = pl->inter;
      p.n_fb = (pl->inter + kHalf - 1) / kHalf;
      p.kblocks = pl->d / kBK;
      p.out = pl->h;
      p.ldo = pl->inter;
    } else {
      maps.w[0] = pl->m_down;
      maps.tok = pl->m_h;
      p.seg_k0[1] = pl->inter;
      p.n_feat = pl->d;
      p.n_fb = (pl->d + 2 * kHalf - 1) / (2 * kHalf);
      p.kblocks = pl->inter / kBK;
      p.out = out;
      p.ldo = pl->d;
    }
    int n;
    const cudaError_t e = launch_tc(maps, p, pass == 0 ? kEpiGlu : kEpiStore, pl->sm_count, st, false, &n);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace lmoe
