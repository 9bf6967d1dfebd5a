// Tensor-core engine of the layer: one persistent, warp-specialised tcgen05 GEMM kernel
// serves every contraction ("Stable LatentMoE": router, down_proj, GroupedExperts gate/up +
// SiTU-GLU, expert down, shared experts, up_proj + shared down), and the dense first-layer
// FFN.  Operands are bf16 (kind::f16), or e4m3 for the fp8 routed experts (kind::f8f6f4).
// The kernel runs either on single CTAs (cta_group::1, M = 128 per MMA) or on pairs of CTAs
// (thread-block clusters of two, cta_group::2, M = 256 per MMA with 128 weight rows and half
// of the tokens in each CTA's shared memory, which halves the token operand each CTA stages
// and its tensor core reads per weight byte; the price is a longer round trip per stage,
// since a stage is consumed only when both CTAs hold it).
//
// Weight-stationary tiles.  Each K step of a tile issues two MMAs against the same tokens:
//   * GLU tiles: the gate rows and the up rows of the same output features, so a TMEM lane
//     holds both branches of one feature and the SiTU-GLU epilogue needs no exchange;
//   * store tiles: two consecutive blocks of output rows (the second is skipped when it lies
//     past the last output row).
// K advances one 128-byte swizzle row at a time (64 bf16 or 128 e4m3 values per stage row);
// each weight stage holds one CTA's 128 rows of one operand (16 KB).
// Token tiles: an expert segment (or the dense batch) is cut into tiles of at most kTokMax
// tokens, N rounded up to 16 per CTA.  Routed token rows are gathered straight from z by the
// slot -> token map (cp.async, 16 bytes per thread, into the swizzled layout), so no
// slot-ordered copy of the rows exists.  Each weight tile is streamed once per token tile (once per expert at prefill
// sizes), and token rows are re-read from L2 by every feature block of their tile.
// Accumulators: TMEM holds 512 fp32 columns in two 256-column slots.  A tile of at most 128
// tokens takes one slot (first MMA in its first 128 columns, second MMA in the second), so two
// such tiles double-buffer; a wider tile takes both slots, and its epilogue packs the results
// into registers and releases TMEM before the global stores.
// Roles (512 threads per CTA): warp 0 streams weight rows, warp 2 streams token rows; warp 1
// issues the MMAs (in a pair: the first CTA's warp 1, which commits each stage back to both
// CTAs' rings, while the second CTA's warp 1 relays "k-block landed" of its own rings to the
// first, so that each CTA's copies complete on its own barriers and each can drain them);
// warps 4-15 drain the accumulators of their own CTA with tcgen05.ld and write the outputs.
// Every mbarrier wait is bounded: on expiry the kernel records the timeout status, tells the
// peer CTA, drains what it issued and returns; a pair meets at a cluster barrier before TMEM
// is freed and the CTAs exit.
#include <cuda.h>
#include <cuda_fp8.h>

#include <cstring>
#include <new>

#include "common.cuh"
#include "gemm_tc.h"

namespace lmoe {
namespace {

constexpr int kBK = 64;                          // bf16 K elements per stage row (128 bytes)
constexpr int kRows = 128;                       // weight rows per CTA per MMA
constexpr int kTokMax = kTileM;                  // tokens per tile (MMA N)
constexpr int kTokBox = 16;                      // token rows per tiled TMA box
constexpr int kHalfBytes = kRows * 128;          // one CTA's 128 rows of one weight operand: 16 KB
constexpr int kWStageBytes = 2 * kHalfBytes;     // one weight stage: both operands of a K step
constexpr int kSlotCols = 256;
constexpr int kEpiWarps = 12;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 128 + kEpiThreads;
constexpr int kMaxChunks = (kTokMax / 32 + 2) / 3;   // 32-token chunks per epilogue warp
constexpr int kSchedMax = 1024;                  // schedule entries kept in shared memory
constexpr int kDenseGroup = 8;                   // token tiles per raster group (dense GEMMs)
constexpr unsigned long long kTimeoutNs = 2000000000ull;    // 2 s per wait
constexpr unsigned long long kInjectTimeoutNs = 20000000ull;  // 20 ms when a timeout is injected
static_assert(kTokMax % 32 == 0 && kTokMax <= 256, "MMA N limit");
// How a tile's token rows reach shared memory: tiled TMA boxes of consecutive rows of the
// token map; TMA tile::gather4 of the rows the slot -> token map names (the map's box one row
// high); or cp.async of those rows, 16 bytes per thread, by warps 2-3.
enum TokMode { kTokTiled = 0, kTokGather4 = 1, kTokCpAsync = 2 };

// Geometry of the single-CTA (CTAS = 1) and pair (CTAS = 2) kernels.
template <int CTAS>
struct Geo {
  static constexpr int kM = kRows * CTAS;               // MMA M
  static constexpr int kGluFeat = kRows * CTAS;         // output features of a GLU tile
  static constexpr int kStoreRows = 2 * kRows * CTAS;   // output rows of a store tile
  static constexpr int kQuant = 16 * CTAS;              // N granularity
  static constexpr int kTokRows = kTokMax / CTAS;       // token rows per CTA and tile
  static constexpr int kTStageBytes = kTokRows * 128;
  static constexpr int kWStages = CTAS == 2 ? 5 : 4;
  static constexpr int kTStages = CTAS == 2 ? 4 : 3;
  static constexpr int kGatherRows = kTokRows / 8;           // cp.async: rows per producer thread and stage
  static constexpr int kGather4 = (kTokRows / 4 + 31) / 32;   // gather4: copies per lane and stage
  // barriers: weight full / empty, token full / empty, peer k-block full (pairs: per token
  // stage, the second CTA's token stage and the weight stages of the same k-block have
  // landed), TMEM full / empty per slot, drain
  static constexpr int kBarWFull = 0, kBarWEmpty = kWStages;
  static constexpr int kBarTFull = 2 * kWStages, kBarTEmpty = kBarTFull + kTStages, kBarTPeer = kBarTFull + 2 * kTStages;
  static constexpr int kBarAFull = kBarTFull + 3 * kTStages, kBarAEmpty = kBarAFull + 2, kBarDrain = kBarAEmpty + 2;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffT = kWStages * kWStageBytes;
  static constexpr int kOffSched = kOffT + kTStages * kTStageBytes;
  static constexpr int kOffBars = kOffSched + 2 * kSchedMax * 4;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = 1024 + kOffMisc + 16;
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  static_assert(kOffT % 1024 == 0 && kTStageBytes % 1024 == 0, "swizzle atoms");
  static_assert(kTokRows % kTokBox == 0 && kTokRows / kTokBox <= 32, "token boxes per stage");
};

struct TcMaps {
  CUtensorMap w[kMaxKSeg];  // weight (MMA A) maps, one per K segment; GLU: w[0] = gate
  CUtensorMap wup;          // GLU up-branch weights
  CUtensorMap tok;          // token (MMA B) rows, 16-row boxes (not used when tokens are gathered)
};

struct TcParams {
  int nseg;
  int seg_k0[kMaxKSeg + 1];
  int seg_row0[kMaxKSeg];
  int w_group_rows;         // weight rows per group (routed experts), 0 for dense
  int n_feat;               // output features
  int n_fb;                 // feature blocks per token tile (store: 2 MMA row blocks, GLU: one)
  int kblocks;              // K / (K elements per stage row)
  int bt;                   // dense: tokens
  int tok_tile;             // dense: tokens per tile (<= kTokMax, multiple of 16 per CTA)
  const int32_t* seg_off;   // grouped: [G + 1] token segments (slots)
  const int32_t* mtile_off; // grouped: [G + 1] prefix of kTokMax-token tiles
  int G;                    // grouped: number of groups, 0 for dense
  int tok_mode;             // token rows: kTokTiled, kTokGather4 or kTokCpAsync
  const int32_t* perm;      // routed experts: slot -> token row (gathers, fp8 token scales)
  const uint8_t* gsrc;      // kTokCpAsync: row 0 of the token rows
  long long gld;            // kTokCpAsync: bytes between rows
  void* out;
  long long ldo;
  float* out_t;
  long long ldt;
  const float* bias;
  float beta, beta_u;
  float inv_beta, inv_beta_u;
  // fp8 (e4m3) routed experts: acc * wscale[row] * tscale[token] is the gate / up value (GLU,
  // up rows scaled by wscale_up), h is stored as e4m3(act * h_mul); the store kind writes
  // acc * wscale[row] * out_mul
  const float* wscale;
  const float* wscale_up;
  const float* tscale;
  float h_mul, out_mul;
  unsigned long long timeout_ns;  // limit of every mbarrier wait
  int inject;               // test hook: the token producers leave their stages unfilled
  uint32_t* status;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
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
// Arrive on a barrier of a CTA of the cluster (address from map_to_rank).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
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

// Abort state of a CTA: its own flag and, in a pair, the address of the peer CTA's flag.
struct Abort {
  volatile int* flag;
  uint32_t peer_flag;
  bool pair;
  uint32_t* status;
  __device__ __forceinline__ void raise(uint32_t bits) const {
    *flag = 1;
    if (pair) asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_flag), "r"(1) : "memory");
    atomicOr(status, bits);
  }
};

// Bounded wait.  Gives up when the deadline passes (raising abort + timeout status) or, if
// honour_abort, as soon as this CTA has been told to abort.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Abort& ab, unsigned long long limit_ns,
                                       bool honour_abort = true) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (honour_abort && *ab.flag) return false;
      if (global_ns() - t0 > limit_ns) {
        ab.raise(kStatusTimeout);
        return false;
      }
    }
  }
}

// 2-D TMA tile load into this CTA's shared memory, completing on its own mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// Four rows y0..y3 of columns [x, x + box) (the map's box is one row high) into 4 consecutive
// 128-byte rows at dst; the map's swizzle applies as for a tiled copy.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2,
                                            int y3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar), "l"(policy)
      : "memory");
}
// 16 bytes global -> shared through L2 (the gathered token rows).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on the barrier once every cp.async this thread issued so far has landed (the barrier
// counts one arrival per producer thread).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Makes shared memory written through the generic proxy (cp.async) visible to the tensor
// core's reads, which go through the async proxy.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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

// tcgen05 instructions of the single-CTA (CTAS = 1) and pair (CTAS = 2) kernels.
template <int CTAS>
struct Tc;

template <>
struct Tc<1> {
  static __device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  static __device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols));
  }
  // Arrive on the barrier once the MMAs this thread issued so far are complete.
  static __device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
  }
  static __device__ __forceinline__ void commit_local(uint32_t bar) { commit(bar); }
  static __device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  }
  static __device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  }
};

template <>
struct Tc<2> {
  static __device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  static __device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols));
  }
  // Arrive on the barrier at this shared-memory offset in both CTAs of the pair once the MMAs
  // this thread issued so far are complete.
  static __device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
  }
  // The same, on this CTA's barrier only.
  static __device__ __forceinline__ void commit_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
  }
  // D[256 x N] (+)= A[256 x K-step] B[K-step x N]: A rows and B columns split over the two
  // CTAs' shared memory at the same offsets, D rows split over the two CTAs' TMEM.
  static __device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  }
  static __device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
  }
};

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

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes
// in 8-row (1024-byte) groups; start address advanced by 32 bytes per K step of 16.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor: fp32 accumulator, A and B K-major; A / B format 1 = bf16 under
// kind::f16, 0 = e4m3 under kind::f8f6f4; N >> 3 and M >> 4.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_e4m3(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
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
  int g, fb, tok0, ntok, ncol;  // ncol: MMA N (ntok rounded up to 16 per CTA)
};

__device__ __forceinline__ int num_tiles(const TcParams& p) {
  if (p.G > 0) return p.mtile_off[p.G] * p.n_fb;
  return ((p.bt + p.tok_tile - 1) / p.tok_tile) * p.n_fb;
}

// Grouped: tiles ordered (expert, feature block, token tile), so the CTAs working at the same
// time share weight rows and token rows in L2; seg/mt are the expert segment and tile
// prefixes (shared memory when they fit).  Dense: token tiles in groups of kDenseGroup,
// feature blocks inside a group.
template <int CTAS>
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
    r.tok0 = seg[lo] + tb * kTokMax;
    r.ntok = min(kTokMax, seg[lo + 1] - r.tok0);
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
  constexpr int q = Geo<CTAS>::kQuant;
  r.ncol = (r.ntok + q - 1) / q * q;
  return r;
}

// K order of a tile: the feature blocks of one token tile run on neighbouring CTAs at the
// same time and read the same token rows, so each starts its K loop at a different offset
// (evenly spread); every token k-block is then fetched from DRAM by one CTA and found in L2
// by the others.  The order is fixed per tile (the same in both CTAs of a pair), so results
// are deterministic.
__device__ __forceinline__ int k_rot(const TcParams& p, const Tile& tl, int kb) {
  int k = kb + (int)(((long long)tl.fb * p.kblocks) / p.n_fb);
  return k >= p.kblocks ? k - p.kblocks : k;
}

// Weight operands (MMAs) per K step: GLU always two (gate, up); store / router one or two
// blocks of output rows.
template <int EPI, int CTAS>
__device__ __forceinline__ int tile_halves(const TcParams& p, const Tile& tl) {
  if (EPI == kEpiGlu) return 2;
  return (p.n_feat - tl.fb * Geo<CTAS>::kStoreRows > Geo<CTAS>::kM) ? 2 : 1;
}

// TMEM columns of the two accumulators of a tile: narrow tiles (<= 128 tokens) use slot s,
// wide ones both slots.
__device__ __forceinline__ uint32_t acc_col(bool wide, int slot, int h) {
  return wide ? (uint32_t)(h * kSlotCols) : (uint32_t)(slot * kSlotCols + h * kRows);
}

// ------------------------------------------------------------------ the kernel
template <int EPI, bool F8, int CTAS>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  using G = Geo<CTAS>;
  constexpr int kBKe = F8 ? 2 * kBK : kBK;   // K elements per stage row (128 bytes)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  const uint32_t wbase = base;
  const uint32_t tbase = base + G::kOffT;
  int32_t* s_seg = reinterpret_cast<int32_t*>(sbase + G::kOffSched);
  int32_t* s_mt = s_seg + kSchedMax;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + G::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(sbase + G::kOffBars);
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CTAS == 2 ? cluster_rank() : 0u;   // rank 0 issues the MMAs
  const int unit = blockIdx.x / CTAS, nunits = gridDim.x / CTAS;
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kWStages; ++s) {
      mbar_init(bar(G::kBarWFull + s), 1);
      mbar_init(bar(G::kBarWEmpty + s), 1);
    }
    for (int s = 0; s < G::kTStages; ++s) {
      mbar_init(bar(G::kBarTFull + s), p.tok_mode == kTokCpAsync ? 64 : 1);   // cp.async: one arrival per producer thread
      mbar_init(bar(G::kBarTEmpty + s), 1);
      mbar_init(bar(G::kBarTPeer + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(G::kBarAFull + a), 1);
      mbar_init(bar(G::kBarAEmpty + a), CTAS * kEpiWarps);   // the epilogue warps of every CTA
    }
    mbar_init(bar(G::kBarDrain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const bool sched_smem = p.G > 0 && p.G < kSchedMax;
  if (sched_smem) {
    for (int i = threadIdx.x; i <= p.G; i += blockDim.x) {
      s_seg[i] = p.seg_off[i];
      s_mt[i] = p.mtile_off[i];
    }
  }
  if (warp == 1) Tc<CTAS>::alloc(smem_u32(tmem_slot), 2 * kSlotCols);
  tc_fence_before();
  __syncthreads();
  if (CTAS == 2) cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t* seg = sched_smem ? s_seg : p.seg_off;
  const int32_t* mt = sched_smem ? s_mt : p.mtile_off;
  const int ntiles = num_tiles(p);
  Abort ab;
  ab.flag = abort_flag;
  ab.pair = CTAS == 2;
  ab.peer_flag = CTAS == 2 ? map_to_rank(smem_u32((const void*)abort_flag), rank ^ 1u) : 0u;
  ab.status = p.status;

  if (warp == 0) {
    // ---------------------------------------------------------------- weight producer
    // Weight operand h of k-block kb of a tile, this CTA's 128 rows: tensor map and coordinates.
    auto w_src = [&](const Tile& tl, int kb, int h, const CUtensorMap*& m, int& x, int& y) {
      const int k = kb * kBKe;
      if (EPI == kEpiGlu) {
        m = h ? &maps.wup : &maps.w[0];
        x = k;
        y = tl.g * p.w_group_rows + tl.fb * G::kGluFeat + (int)rank * kRows;
      } else {
        int s = 0;
#pragma unroll
        for (int i = 1; i < kMaxKSeg; ++i)
          if (i < p.nseg && k >= p.seg_k0[i]) s = i;
        m = &maps.w[s];
        x = k - p.seg_k0[s];
        y = p.seg_row0[s] + tl.g * p.w_group_rows + tl.fb * G::kStoreRows + h * G::kM + (int)rank * kRows;
      }
    };
    if (lane == 0) {
      const uint64_t wpol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0, pending = 0, pend_parity = 0;
      bool stop = false;
      for (int t = unit; t < ntiles && !stop; t += nunits) {
        const Tile tl = decode_tile<CTAS>(p, seg, mt, t);
        const int nh = tile_halves<EPI, CTAS>(p, tl);
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(bar(G::kBarWEmpty + stage), phase ^ 1u, ab, p.timeout_ns)) { stop = true; break; }
          pending &= ~(1u << stage);
          mbar_expect_tx(bar(G::kBarWFull + stage), (uint32_t)(nh * kHalfBytes));
          const int kr = k_rot(p, tl, kb);
          for (int h = 0; h < nh; ++h) {
            const CUtensorMap* m;
            int x, y;
            w_src(tl, kr, h, m, x, y);
            tma_load_2d(wbase + stage * kWStageBytes + h * kHalfBytes, m, x, y, bar(G::kBarWFull + stage), wpol);
          }
          pending |= 1u << stage;
          pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == G::kWStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (stop) {
        // no copy may still be landing in shared memory when the block exits
        for (int s = 0; s < G::kWStages; ++s)
          if (pending & (1u << s)) mbar_wait(bar(G::kBarWFull + s), (pend_parity >> s) & 1u, ab, p.timeout_ns, false);
      }
    }
    __syncwarp();
  } else if (warp == 2 && p.tok_mode != kTokCpAsync) {
    // ---------------------------------------------------------------- token producer (TMA)
    const uint64_t tpol = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, pending = 0, pend_parity = 0;
    bool stop = false;
    for (int t = unit; t < ntiles && !stop; t += nunits) {
      const Tile tl = decode_tile<CTAS>(p, seg, mt, t);
      const int rows = tl.ncol / CTAS;               // this CTA's token rows: [r0, r0 + rows)
      const int r0 = tl.tok0 + (int)rank * rows;
      // gather4: this lane's slots -> token rows (rows past the tile read token 0; their columns
      // are never stored)
      int gy[G::kGather4][4];
#pragma unroll
      for (int c = 0; c < G::kGather4; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = (lane + 32 * c) * 4 + i, sl = r0 + rr;
          gy[c][i] = (p.tok_mode == kTokGather4 && rr < rows && sl < tl.tok0 + tl.ntok) ? p.perm[sl] : 0;
        }
      for (int kb = 0; kb < p.kblocks; ++kb) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(bar(G::kBarTEmpty + stage), phase ^ 1u, ab, p.timeout_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) { stop = true; break; }
        pending &= ~(1u << stage);
        if (p.inject) {
          // test hook: nothing fills this stage, so its consumers' bounded waits run out
          if (++stage == G::kTStages) { stage = 0; phase ^= 1u; }
          continue;
        }
        if (lane == 0) mbar_expect_tx(bar(G::kBarTFull + stage), (uint32_t)rows * 128u);
        __syncwarp();
        const uint32_t dst = tbase + stage * G::kTStageBytes;
        const int x = k_rot(p, tl, kb) * kBKe;
        if (p.tok_mode == kTokGather4) {
#pragma unroll
          for (int c = 0; c < G::kGather4; ++c) {
            const int quad = lane + 32 * c;
            if (quad * 4 < rows)
              tma_gather4(dst + quad * 512, &maps.tok, x, gy[c][0], gy[c][1], gy[c][2], gy[c][3],
                          bar(G::kBarTFull + stage), tpol);
          }
        } else if (lane < rows / kTokBox) {
          tma_load_2d(dst + lane * (kTokBox * 128), &maps.tok, x, r0 + lane * kTokBox, bar(G::kBarTFull + stage), tpol);
        }
        pending |= 1u << stage;
        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == G::kTStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (stop && lane == 0) {
      for (int s = 0; s < G::kTStages; ++s)
        if (pending & (1u << s)) mbar_wait(bar(G::kBarTFull + s), (pend_parity >> s) & 1u, ab, p.timeout_ns, false);
    }
    __syncwarp();
  } else if ((warp == 2 || warp == 3) && p.tok_mode == kTokCpAsync) {
    // ---------------------------------------------------------------- token producer (gather)
    // Routed token rows straight from the token matrix through the slot -> token map: warps 2-3
    // copy 16-byte chunks with cp.async (a warp instruction covers four 128-byte rows) into the
    // 128-byte-swizzled layout the MMA reads (chunk c of row r at r * 128 + (c ^ (r % 8)) * 16).
    const int pt = threadIdx.x - 64;                 // 0..63
    const int chunk = pt & 7, rsub = pt >> 3;        // this thread: chunk `chunk` of rows rsub + 8 j
    const uint32_t swz = (uint32_t)((chunk ^ rsub) * 16) + (uint32_t)rsub * 128u;
    const int esz = F8 ? 1 : 2;
    int stage = 0;
    uint32_t phase = 0, pending = 0, pend_parity = 0;
    bool stop = false;
    for (int t = unit; t < ntiles && !stop; t += nunits) {
      const Tile tl = decode_tile<CTAS>(p, seg, mt, t);
      const int rows = tl.ncol / CTAS;               // this CTA's token rows: [r0, r0 + rows)
      const int r0 = tl.tok0 + (int)rank * rows;
      // source row of each of this thread's rows (rows past the tile read row 0; their columns
      // are never stored)
      const uint8_t* src[G::kGatherRows];
#pragma unroll
      for (int j = 0; j < G::kGatherRows; ++j) {
        const int rr = rsub + 8 * j, sl = r0 + rr;
        const int tok = (rr < rows && sl < tl.tok0 + tl.ntok) ? p.perm[sl] : 0;
        src[j] = p.gsrc + (long long)tok * p.gld + chunk * 16;
      }
      for (int kb = 0; kb < p.kblocks; ++kb) {
        bool ok = true;
        if (pt == 0) ok = mbar_wait(bar(G::kBarTEmpty + stage), phase ^ 1u, ab, p.timeout_ns);
        if (named_sync_or(2, 64, !ok)) { stop = true; break; }
        pending &= ~(1u << stage);
        if (p.inject) {
          // test hook: nothing fills this stage, so its consumers' bounded waits run out
          if (++stage == G::kTStages) { stage = 0; phase ^= 1u; }
          continue;
        }
        const uint32_t dst = tbase + stage * G::kTStageBytes + swz;
        const long long col = (long long)k_rot(p, tl, kb) * kBKe * esz;
#pragma unroll
        for (int j = 0; j < G::kGatherRows; ++j)
          if (rsub + 8 * j < rows) cp_async16(dst + (uint32_t)j * 1024u, src[j] + col);
        cp_async_arrive(bar(G::kBarTFull + stage));
        pending |= 1u << stage;
        pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == G::kTStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (stop) {
      // no copy may still be landing in shared memory when the block exits
      cp_async_wait_all();
      named_sync_or(2, 64, false);
      if (pt == 0)
        for (int s = 0; s < G::kTStages; ++s)
          if (pending & (1u << s)) mbar_wait(bar(G::kBarTFull + s), (pend_parity >> s) & 1u, ab, p.timeout_ns, false);
    }
  } else if (warp == 1 && rank == 1) {
    // ---------------------------------------------------------------- relay (second CTA of a pair)
    // Tells the first CTA, k-block by k-block in consumption order, that this CTA's weight
    // and token stages of the k-block have landed (one arrival per k-block).
    if (lane == 0) {
      int ws = 0, ts = 0;
      uint32_t wph = 0, tph = 0;
      bool stop = false;
      for (int t = unit; t < ntiles && !stop; t += nunits) {
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(bar(G::kBarWFull + ws), wph, ab, p.timeout_ns) ||
              !mbar_wait(bar(G::kBarTFull + ts), tph, ab, p.timeout_ns)) { stop = true; break; }
          if (++ws == G::kWStages) { ws = 0; wph ^= 1u; }
          if (p.tok_mode == kTokCpAsync) fence_proxy_async();
          mbar_arrive_cluster(map_to_rank(bar(G::kBarTPeer + ts), 0));
          if (++ts == G::kTStages) { ts = 0; tph ^= 1u; }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int ws = 0, ts = 0, slot = 0;
      uint32_t wph = 0, tph = 0;
      uint32_t aph[2] = {0u, 0u};
      bool stop = false, issued = false;
      for (int t = unit; t < ntiles && !stop; t += nunits) {
        const Tile tl = decode_tile<CTAS>(p, seg, mt, t);
        const bool wide = tl.ncol > kRows;
        const int nh = tile_halves<EPI, CTAS>(p, tl);
        const uint32_t idesc = F8 ? idesc_e4m3(G::kM, tl.ncol) : idesc_bf16(G::kM, tl.ncol);
        if (wide) {
          if (!mbar_wait(bar(G::kBarAEmpty + 0), aph[0] ^ 1u, ab, p.timeout_ns) ||
              !mbar_wait(bar(G::kBarAEmpty + 1), aph[1] ^ 1u, ab, p.timeout_ns)) { stop = true; break; }
        } else {
          if (!mbar_wait(bar(G::kBarAEmpty + slot), aph[slot] ^ 1u, ab, p.timeout_ns)) { stop = true; break; }
        }
        tc_fence_after();
        for (int kb = 0; kb < p.kblocks && !stop; ++kb) {
          if (!mbar_wait(bar(G::kBarWFull + ws), wph, ab, p.timeout_ns) ||
              !mbar_wait(bar(G::kBarTFull + ts), tph, ab, p.timeout_ns) ||
              (CTAS == 2 && !mbar_wait(bar(G::kBarTPeer + ts), tph, ab, p.timeout_ns))) { stop = true; break; }
          if (p.tok_mode == kTokCpAsync) fence_proxy_async();
          tc_fence_after();
          const uint64_t bd = smem_desc(tbase + ts * G::kTStageBytes);
          for (int h = 0; h < nh; ++h) {
            const uint64_t ad = smem_desc(wbase + ws * kWStageBytes + h * kHalfBytes);
            const uint32_t d = tmem_base + acc_col(wide, slot, h);
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j) {
              if (F8) Tc<CTAS>::mma_f8(d, ad + 2u * j, bd + 2u * j, idesc, (kb | j) != 0 ? 1u : 0u);
              else Tc<CTAS>::mma_bf16(d, ad + 2u * j, bd + 2u * j, idesc, (kb | j) != 0 ? 1u : 0u);
            }
          }
          issued = true;
          Tc<CTAS>::commit(bar(G::kBarWEmpty + ws));
          if (++ws == G::kWStages) { ws = 0; wph ^= 1u; }
          Tc<CTAS>::commit(bar(G::kBarTEmpty + ts));
          if (++ts == G::kTStages) { ts = 0; tph ^= 1u; }
        }
        if (stop) break;
        if (wide) {
          Tc<CTAS>::commit(bar(G::kBarAFull + 0));
          Tc<CTAS>::commit(bar(G::kBarAFull + 1));
          aph[0] ^= 1u;
          aph[1] ^= 1u;
        } else {
          Tc<CTAS>::commit(bar(G::kBarAFull + slot));
          aph[slot] ^= 1u;
          slot ^= 1;
        }
      }
      if (stop && issued) {
        // every MMA issued reads shared memory (of both CTAs of a pair) and writes TMEM: wait
        // for them before the block can exit
        Tc<CTAS>::commit_local(bar(G::kBarDrain));
        mbar_wait(bar(G::kBarDrain), 0, ab, p.timeout_ns, false);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int sub = (warp - 4) >> 2;        // which 32-token chunks: sub, sub + 3, ...
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t aempty[2] = {bar(G::kBarAEmpty + 0), bar(G::kBarAEmpty + 1)};
    if (CTAS == 2) {
      aempty[0] = map_to_rank(aempty[0], 0);
      aempty[1] = map_to_rank(aempty[1], 0);
    }
    int slot = 0;
    uint32_t aph[2] = {0u, 0u};
    for (int t = unit; t < ntiles; t += nunits) {
      const Tile tl = decode_tile<CTAS>(p, seg, mt, t);
      const bool wide = tl.ncol > kRows;
      const int nh = tile_halves<EPI, CTAS>(p, tl);
      bool ok;
      if (wide) ok = mbar_wait(bar(G::kBarAFull + 0), aph[0], ab, p.timeout_ns) &&
                     mbar_wait(bar(G::kBarAFull + 1), aph[1], ab, p.timeout_ns);
      else ok = mbar_wait(bar(G::kBarAFull + slot), aph[slot], ab, p.timeout_ns);
      if (named_sync_or(1, kEpiThreads, !ok || *abort_flag)) break;
      tc_fence_after();
      const uint32_t c0 = lane_base + acc_col(wide, slot, 0);
      const uint32_t c1 = lane_base + acc_col(wide, slot, 1);
      const int nchunks = (tl.ntok + 31) >> 5;
      // this lane's output features: GLU fo, store fo + h * kM
      const int fo = (EPI == kEpiGlu ? tl.fb * G::kGluFeat : tl.fb * G::kStoreRows) + (int)rank * kRows + q * 32 + lane;
      // Results of this warp's chunks (<= kMaxChunks), packed bf16 pairs of consecutive
      // tokens (e4m3 quads for the fp8 GLU); TMEM is released before they are written out.
      uint32_t res[kMaxChunks][2][16];
      if (EPI == kEpiGlu) {
        // fp8: the gate and up row scales of this lane's feature
        float sg = 1.f, su = 1.f;
        if (F8 && fo < p.n_feat) {
          sg = p.wscale[(long long)tl.g * p.w_group_rows + fo];
          su = p.wscale_up[(long long)tl.g * p.w_group_rows + fo];
        }
#pragma unroll
        for (int ci = 0; ci < kMaxChunks; ++ci) {
          const int c = sub + 3 * ci;
          if (c < nchunks) {
            uint32_t g[32], u[32];
            tmem_ld32(c0 + c * 32, g);
            tmem_ld32(c1 + c * 32, u);
            float ts = 1.f;   // fp8: this lane's token scale (lane j holds token j of the chunk)
            if (F8 && c * 32 + lane < tl.ntok) {
              const int slot_ix = tl.tok0 + c * 32 + lane;
              ts = p.tscale[p.perm ? p.perm[slot_ix] : slot_ix];
            }
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
                res[ci][0][j >> 2] = word;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                res[ci][0][j] = pack_bf16x2(situ_glu_fast(__uint_as_float(g[2 * j]), __uint_as_float(u[2 * j]), p),
                                            situ_glu_fast(__uint_as_float(g[2 * j + 1]), __uint_as_float(u[2 * j + 1]), p));
            }
          }
        }
      } else if (EPI == kEpiStore) {
#pragma unroll
        for (int ci = 0; ci < kMaxChunks; ++ci) {
          const int c = sub + 3 * ci;
          if (c < nchunks) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (h < nh) {
                uint32_t v[32];
                tmem_ld32((h ? c1 : c0) + c * 32, v);
                float sc = 1.f;   // fp8: row scale times the activation scale
                if (F8) {
                  const int fh = fo + h * G::kM;
                  if (fh < p.n_feat) sc = p.wscale[(long long)tl.g * p.w_group_rows + fh] * p.out_mul;
                }
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  res[ci][h][j] = pack_bf16x2(__uint_as_float(v[2 * j]) * sc, __uint_as_float(v[2 * j + 1]) * sc);
              }
            }
          }
        }
      } else {
        // router: fp32 logits and their transpose, written straight from TMEM
        for (int c = sub; c < nchunks; c += 3) {
          const int nj = min(32, tl.ntok - c * 32);
          for (int h = 0; h < nh; ++h) {
            uint32_t v[32];
            tmem_ld32((h ? c1 : c0) + c * 32, v);
            tmem_wait_ld();
            const int fout = fo + h * G::kM;
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
        auto arrive = [&](int a) {
          if (CTAS == 2) mbar_arrive_cluster(aempty[a]);
          else mbar_arrive(aempty[a]);
        };
        if (wide) { arrive(0); arrive(1); }
        else arrive(slot);
      }
      if (EPI != kEpiRouter) {
#pragma unroll
        for (int ci = 0; ci < kMaxChunks; ++ci) {
          const int c = sub + 3 * ci;
          if (c >= nchunks) continue;
          const int nj = min(32, tl.ntok - c * 32);
#pragma unroll
          for (int h = 0; h < (EPI == kEpiGlu ? 1 : 2); ++h) {
            const int fout = fo + h * G::kM;
            if (h >= nh || fout >= p.n_feat) continue;
            if (F8 && EPI == kEpiGlu) {
              uint8_t* o = static_cast<uint8_t*>(p.out) + (long long)(tl.tok0 + c * 32) * p.ldo + fout;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nj) o[(long long)j * p.ldo] = (uint8_t)(res[ci][0][j >> 2] >> (8 * (j & 3)));
            } else {
              bf16* o = static_cast<bf16*>(p.out) + (long long)(tl.tok0 + c * 32) * p.ldo + fout;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nj) {
                  const uint32_t w2 = res[ci][h][j >> 1];
                  o[(long long)j * p.ldo] = __ushort_as_bfloat16((unsigned short)((j & 1) ? (w2 >> 16) : (w2 & 0xffffu)));
                }
            }
          }
        }
      }
      if (wide) { aph[0] ^= 1u; aph[1] ^= 1u; }
      else { aph[slot] ^= 1u; slot ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (CTAS == 2) cluster_sync();  // no copy, MMA or remote arrive of either CTA is still pending
  tc_fence_after();
  if (warp == 1) Tc<CTAS>::dealloc(tmem_base, 2 * kSlotCols);
}

// Routed token rows in slot order: zp[slot] = rows[perm[slot]]; one warp per row, 16-byte
// vectors (each row is read from L2-resident rows and written once).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ rows, const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ offsets, int n_experts,
                                                          int vec_per_row, uint4* __restrict__ zp) {
  const int nslots = offsets[n_experts];
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int slot = blockIdx.x * wpb + (threadIdx.x >> 5); slot < nslots; slot += gridDim.x * wpb) {
    const uint4* src = rows + (long long)perm[slot] * vec_per_row;
    uint4* dst = zp + (long long)slot * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) dst[v] = src[v];
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

// Token tile of a dense GEMM: the multiple of quant in [128, kTokMax] that minimises
// waves x (tile + a fixed per-tile cost of 32 tokens) over the persistent units, so the last
// wave is nearly full (e.g. the 8192-token router: 172 tiles of 192 tokens leave most of a
// second wave idle; 256 tiles of 128 fill it, and narrow tiles double-buffer TMEM).
int dense_tok_tile(int bt, int n_fb, int units, int quant) {
  int best = kTokMax;
  long long best_cost = -1;
  for (int tt = kTokMax; tt >= 128; tt -= quant) {
    const long long tiles = (long long)((bt + tt - 1) / tt) * n_fb;
    const long long waves = (tiles + units - 1) / units;
    const long long cost = waves * (tt + 32);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = tt; }
  }
  return best;
}

template <int EPI, bool F8, int CTAS>
cudaError_t launch_units(const TcMaps& maps, const TcParams& p, int units, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(CTAS * units, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Geo<CTAS>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CTAS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CTAS == 2 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<EPI, F8, CTAS>, maps, p);
}

template <int CTAS>
cudaError_t prepare_mode(bool f8) {
  const int smem = Geo<CTAS>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<kEpiStore, false, CTAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_kernel<kEpiGlu, false, CTAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_gemm_kernel<kEpiRouter, false, CTAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && f8)
    e = cudaFuncSetAttribute(tc_gemm_kernel<kEpiGlu, true, CTAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && f8)
    e = cudaFuncSetAttribute(tc_gemm_kernel<kEpiStore, true, CTAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

cudaError_t prepare_all(bool f8) {
  cudaError_t e = prepare_mode<1>(f8);
  return e == cudaSuccess ? prepare_mode<2>(f8) : e;
}

// Pairs that can be resident at once, from the occupancy of one cluster of two 512-thread
// CTAs with the pair kernel's shared memory; never more than sm_count / 2.
int resident_pairs(int sm_count) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Geo<2>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<kEpiStore, false, 2>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sm_count / 2;
  }
  return n < sm_count / 2 ? n : sm_count / 2;
}

// One launch of the persistent kernel in the given mode: one CTA (or pair) per resident slot,
// fewer when a dense GEMM has fewer tiles.
template <int CTAS>
cudaError_t launch_mode(const TcMaps& maps, TcParams& p, int epi, int units, cudaStream_t st, bool f8) {
  if (p.G == 0) p.tok_tile = dense_tok_tile(p.bt, p.n_fb, units, Geo<CTAS>::kQuant);
  if (p.G == 0) {
    const long long tiles = (long long)((p.bt + p.tok_tile - 1) / p.tok_tile) * p.n_fb;
    if (tiles < units) units = (int)tiles;
  }
  if (units <= 0) return cudaSuccess;
  if (f8) {
    if (epi == kEpiGlu) return launch_units<kEpiGlu, true, CTAS>(maps, p, units, st);
    return launch_units<kEpiStore, true, CTAS>(maps, p, units, st);
  }
  switch (epi) {
    case kEpiStore: return launch_units<kEpiStore, false, CTAS>(maps, p, units, st);
    case kEpiGlu: return launch_units<kEpiGlu, false, CTAS>(maps, p, units, st);
    default: return launch_units<kEpiRouter, false, CTAS>(maps, p, units, st);
  }
}

// Feature blocks of an output of n features in a mode.
int feature_blocks(int n, int epi, int ctas) {
  const int per = epi == kEpiGlu ? kRows * ctas : 2 * kRows * ctas;
  return (n + per - 1) / per;
}

}  // namespace

// How the routed gate/up GEMM gets its token rows (TokMode).
constexpr int kGateUpTokMode = kTokTiled;

// Mode of each contraction: 2 = CTA pairs, 1 = single CTAs.
constexpr int kOpCtas[kNumOps] = {
    1,  // kOpRouter
    1,  // kOpDown
    1,  // kOpExpertGateUp
    1,  // kOpExpertDown
    1,  // kOpSharedGateUp
    1,  // kOpFinal
};
constexpr int kFfnCtas = 2;

struct TcPlan {
  lmoe_config cfg;
  int max_bt;
  int sm_count;
  int pairs;                                                // resident CTA pairs
  TcBuffers buf;
  bool f8;                                                  // e4m3 routed experts
  CUtensorMap m_gate8, m_up8, m_edown8, m_h8, m_zp8, m_zq8; // their weights, h, token rows
  const float *s_gate, *s_up, *s_down;                      // per-row weight scales
  float h_mul, h_scale;                                     // fixed activation scale (SiTU-GLU bound)
  bool inject;                                              // test hook armed for the next expert gate/up
  CUtensorMap m_router, m_down, m_gate, m_up, m_edown, m_shg, m_shu, m_wup, m_shd;  // weights
  CUtensorMap m_h, m_cat, m_zp, m_zg;                                                 // workspace
};

lmoe_status tc_plan_create(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_fp8_experts* f8, int max_bt,
                           int sm_count, const TcBuffers& buf, TcPlan** plan) {
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
  pl->f8 = f8 != nullptr;
  bool ok = make_map(&pl->m_router, w->w_router, E, d, d, kRows) && make_map(&pl->m_down, w->w_down, L, d, d, kRows);
  if (pl->f8) {
    ok = ok && make_map(&pl->m_gate8, f8->exp_gate, E * I, L, L, kRows, true) &&
         make_map(&pl->m_up8, f8->exp_up, E * I, L, L, kRows, true) &&
         make_map(&pl->m_edown8, f8->exp_down, E * L, I, I, kRows, true) &&
         make_map(&pl->m_h8, buf.h, slots, I, I, kTokBox, true) && make_map(&pl->m_zp8, buf.zp, slots, L, L, kTokBox, true) &&
         make_map(&pl->m_zq8, buf.zq, max_bt, L, L, 1, true);
    pl->s_gate = f8->gate_scale;
    pl->s_up = f8->up_scale;
    pl->s_down = f8->down_scale;
    const float bound = c.beta * c.beta_u;   // |SiTU-GLU| < beta * beta_u
    pl->h_mul = 448.0f / bound;
    pl->h_scale = bound / 448.0f;
  } else {
    ok = ok && make_map(&pl->m_gate, w->exp_gate, E * I, L, L, kRows) && make_map(&pl->m_up, w->exp_up, E * I, L, L, kRows) &&
         make_map(&pl->m_edown, w->exp_down, E * L, I, I, kRows);
  }
  ok = ok && make_map(&pl->m_shg, w->sh_gate, S * Is, d, d, kRows) && make_map(&pl->m_shu, w->sh_up, S * Is, d, d, kRows) &&
       make_map(&pl->m_wup, w->w_up, d, L, L, kRows) && make_map(&pl->m_shd, w->sh_down, S * d, Is, Is, kRows) &&
       make_map(&pl->m_h, buf.h, slots, I, I, kTokBox) && make_map(&pl->m_zp, buf.zp, slots, L, L, kTokBox) &&
       make_map(&pl->m_zg, buf.z, max_bt, L, L, 1) &&
       make_map(&pl->m_cat, buf.cat, max_bt, ldc, ldc, kTokBox);
  if (!ok) {
    delete pl;
    return LMOE_ERR_CUDA;
  }
  if (prepare_all(pl->f8) != cudaSuccess) {
    cudaGetLastError();
    delete pl;
    return LMOE_ERR_CUDA;
  }
  pl->pairs = resident_pairs(sm_count);
  *plan = pl;
  return LMOE_OK;
}

void tc_plan_destroy(TcPlan* plan) { delete plan; }

void tc_inject_wait_timeout(TcPlan* plan) { plan->inject = true; }

int tc_launches(int op, bool f8) {
  if (op != kOpExpertGateUp) return 1;
  return 1 + (f8 ? 1 : 0) + (kGateUpTokMode == kTokTiled ? 1 : 0);
}

cudaError_t launch_gemm_tc(TcPlan* pl, const GemmArgs& a, cudaStream_t st) {
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
  p.tok_tile = kTokMax;
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
      p.perm = a.a_rows;
      p.tok_mode = kGateUpTokMode;
      p.w_group_rows = c.expert_inter;
      p.seg_off = a.seg_off;
      p.mtile_off = a.mtile_off;
      p.G = a.G;
      // the experts' token rows: z, or its per-token e4m3 copy (scale per token)
      const void* rows = pl->buf.z;
      long long row_bytes = (long long)c.latent * 2;
      if (pl->f8) {
        cudaError_t e = launch_quantize_rows(pl->buf.z, a.bt_tokens, c.latent, pl->buf.zq, pl->buf.tscale,
                                             pl->sm_count * 8, st);
        if (e != cudaSuccess) return e;
        rows = pl->buf.zq;
        row_bytes = c.latent;
        maps.w[0] = pl->m_gate8;
        maps.wup = pl->m_up8;
        maps.tok = kGateUpTokMode == kTokTiled ? pl->m_zp8 : pl->m_zq8;
        p.wscale = pl->s_gate;
        p.wscale_up = pl->s_up;
        p.tscale = pl->buf.tscale;
        p.h_mul = pl->h_mul;
        p.kblocks = a.K / (2 * kBK);
        f8 = true;
      } else {
        maps.w[0] = pl->m_gate;
        maps.wup = pl->m_up;
        maps.tok = kGateUpTokMode == kTokTiled ? pl->m_zp : pl->m_zg;
      }
      p.gsrc = static_cast<const uint8_t*>(rows);
      p.gld = row_bytes;
      if (kGateUpTokMode == kTokTiled) {
        // token rows of each expert segment, gathered once into slot order
        gather_rows_kernel<<<pl->sm_count * 8, 256, 0, st>>>(static_cast<const uint4*>(rows), a.a_rows, a.seg_off, a.G,
                                                             (int)(row_bytes / 16), static_cast<uint4*>(pl->buf.zp));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      break;
    }
    case kOpExpertDown:
      if (pl->f8) {
        maps.w[0] = pl->m_edown8;
        maps.tok = pl->m_h8;
        p.wscale = pl->s_down;
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
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  const int ctas = kOpCtas[a.op];
  p.n_fb = feature_blocks(a.N, epi, ctas);
  if (ctas == 2) return launch_mode<2>(maps, p, epi, pl->pairs, st, f8);
  return launch_mode<1>(maps, p, epi, pl->sm_count, st, f8);
}

// ------------------------------------------------------------------ dense SiTU-GLU FFN
struct TcFfnPlan {
  int d, inter, sm_count, pairs;
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
  const bool ok = make_map(&pl->m_gate, w_gate, inter, d, d, kRows) && make_map(&pl->m_up, w_up, inter, d, d, kRows) &&
                  make_map(&pl->m_down, w_down, d, inter, inter, kRows) &&
                  make_map(&pl->m_h, h, max_bt, inter, inter, kTokBox);
  cudaError_t e = ok ? prepare_all(false) : cudaErrorInvalidValue;
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete pl;
    return LMOE_ERR_CUDA;
  }
  pl->pairs = resident_pairs(sm_count);
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
    const int epi = pass == 0 ? kEpiGlu : kEpiStore;
    if (pass == 0) {
      maps.w[0] = pl->m_gate;
      maps.wup = pl->m_up;
      if (!make_map(&maps.tok, x, bt, pl->d, pl->d, kTokBox)) return cudaErrorInvalidValue;
      p.seg_k0[1] = pl->d;
      p.n_feat = pl->inter;
      p.kblocks = pl->d / kBK;
      p.out = pl->h;
      p.ldo = pl->inter;
    } else {
      maps.w[0] = pl->m_down;
      maps.tok = pl->m_h;
      p.seg_k0[1] = pl->inter;
      p.n_feat = pl->d;
      p.kblocks = pl->inter / kBK;
      p.out = out;
      p.ldo = pl->d;
    }
    p.n_fb = feature_blocks(p.n_feat, epi, kFfnCtas);
    const cudaError_t e = launch_mode<kFfnCtas>(maps, p, epi, pl->pairs, st, false);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace lmoe
