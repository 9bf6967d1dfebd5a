// C ABI of the Stable LatentMoE layer forward: argument validation, the workspace, and the
// launch sequence of the layer ("KimiK3的StableLatentMoE架构解析", ¶"具体前向流程" / Fig. 2:
// router -> down_proj -> GroupedExperts -> latent_norm + weighted fusion -> up_proj, plus the
// shared SiTU-GLU branch on the flattened input).
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/lmoe.h"
#include "common.cuh"
#include "gemm_tc.h"
#include "internal.h"

using namespace lmoe;

struct lmoe_ctx {
  lmoe_config cfg;
  lmoe_weights w;
  int max_bt;
  int device;
  int sm_count;
  cudaStream_t stream;
  bool bf16;
  size_t esz;
  bool check;
  bool use_tc;
  bool f8;              // e4m3 routed experts
  int last_bt;
  double momentum;      // streaming cutoffs: weight of the previous call's cutoff (0 = per call)
  bool state_valid;     // a call has stored its cutoff since momentum was set
  bool norm_sum;        // latent RMSNorm on the weighted sum instead of each expert row
  // workspace (one allocation)
  char* ws;
  size_t ws_bytes;
  float* logits;
  float* logits_t;
  double* alpha;
  double* alpha_state;
  int32_t* idx;
  float* wk;
  int32_t* block_cnt;
  int32_t* counts;
  int32_t* offsets;
  int32_t* mtile_off;
  int32_t* perm;
  int32_t* inv;
  int32_t* topk_list;   // [max_bt + 1] tokens left to the general top-K kernel, then their count
  void* z;
  void* zq;             // fp8 experts: e4m3 rows of z
  void* zp;             // routed token rows in slot order
  void* h;
  void* y;
  void* cat;
  float* tscale;
  float* part;          // split-K partials of the dense GEMMs (bf16 engine)
  uint32_t* status;
  TcPlan* tc;
  // per-stage profiling
  bool prof_on;
  int prof_calls;
  std::vector<cudaEvent_t> prof_ev;   // [kProfCap][LMOE_NUM_STAGES + 1]
  long long launches;
  long long prof_launch_base;
  // host-buffer entry point (created by its first call)
  char* host_ws;               // staging buffers x[0], x[1], out[0], out[1], [max_bt, d] each
  cudaStream_t host_in_st;     // input copies
  cudaStream_t host_run_st;    // forwards of host-buffer calls
  cudaStream_t host_out_st;    // output copies
  cudaEvent_t host_in[2];      // input copy into x[b] done
  cudaEvent_t host_run[2];     // forward of the call that used x[b] and out[b] done
  cudaEvent_t host_out[2];     // output copy from out[b] done
  cudaEvent_t host_last_run;   // the last host-buffer forward done
  cudaEvent_t host_dev_done;   // the last device-buffer call's work done
  int host_next;
  int nvtx_open;             // NVTX ranges this forward has pushed and not yet popped
};

namespace {

constexpr int kProfCap = 1024;

void prof_mark(lmoe_ctx* ctx, int boundary, cudaStream_t st) {
  if (!ctx->prof_on || ctx->prof_calls >= kProfCap) return;
  cudaEventRecord(ctx->prof_ev[(size_t)ctx->prof_calls * (LMOE_NUM_STAGES + 1) + boundary], st);
}

// NVTX ranges of a forward: "lmoe_forward" around the call, one range per stage inside it
// (host-side annotations that profilers align with the kernels each stage launches).
const char* const kStageNames[LMOE_NUM_STAGES] = {
    "router GEMM", "cutoff + top-K + segments", "W_down GEMM", "token gather", "expert gate/up GEMM",
    "expert down GEMM", "RMSNorm + combine", "shared gate/up GEMM", "W_up + shared down GEMM"};

void nvtx_stage(lmoe_ctx* ctx, int boundary) {
  if (ctx->nvtx_open == 0) return;        // not inside lmoe_forward (e.g. lmoe_route)
  if (ctx->nvtx_open > 1) {
    nvtxRangePop();
    --ctx->nvtx_open;
  }
  if (boundary < LMOE_NUM_STAGES) {
    nvtxRangePushA(kStageNames[boundary]);
    ++ctx->nvtx_open;
  }
}

void nvtx_end(lmoe_ctx* ctx) {
  for (; ctx->nvtx_open > 0; --ctx->nvtx_open) nvtxRangePop();
}

// Stage boundary b of a forward: stage b-1 ends and stage b begins.
void stage_mark(lmoe_ctx* ctx, int boundary, cudaStream_t st) {
  prof_mark(ctx, boundary, st);
  nvtx_stage(ctx, boundary);
}

// LMOE_LOG=1: one line on stderr for every failing call of the public API.
lmoe_status logged(const char* fn, lmoe_status s) {
  if (s != LMOE_OK) {
    const char* v = getenv("LMOE_LOG");
    if (v && v[0] == '1') fprintf(stderr, "lmoe: %s: %s\n", fn, lmoe_status_string(s));
  }
  return s;
}

// Test hook: the next workspace / staging allocation of the library fails (lmoe_debug_fail_next_alloc).
std::atomic<int> g_fail_next_alloc{0};

cudaError_t ws_malloc(void** p, size_t bytes) {
  if (g_fail_next_alloc.exchange(0)) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lmoe_status check_cfg(const lmoe_config* c) {
  if (!c) return LMOE_ERR_INVALID_ARG;
  if (c->d <= 0 || c->latent <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->expert_inter <= 0 ||
      c->n_shared <= 0 || c->shared_inter <= 0)
    return LMOE_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts) return LMOE_ERR_INVALID_ARG;
  if (c->dtype != LMOE_F32 && c->dtype != LMOE_BF16) return LMOE_ERR_INVALID_ARG;
  if (!(c->beta > 0.f) || !(c->beta_u > 0.f) || !(c->rms_eps >= 0.f) || c->beta > 3.0e38f ||
      c->beta_u > 3.0e38f || c->rms_eps > 3.0e38f)
    return LMOE_ERR_INVALID_ARG;
  if (c->n_experts > kMaxExperts || c->top_k > kMaxTopK || c->n_shared > kMaxShared)
    return LMOE_ERR_UNSUPPORTED;
  if (c->dtype == LMOE_BF16) {
    if (c->d % 64 || c->latent % 64 || c->expert_inter % 64 || c->shared_inter % 64)
      return LMOE_ERR_UNSUPPORTED;
  } else {
    if (c->latent % 4 || c->shared_inter % 4) return LMOE_ERR_UNSUPPORTED;
  }
  // int32 element offsets inside one weight matrix / row must not overflow
  const long long big = (long long)c->n_experts * c->expert_inter * c->latent;
  if (big >= (1LL << 40)) return LMOE_ERR_UNSUPPORTED;
  return LMOE_OK;
}

lmoe_status check_device_ptr(const void* p) {
  if (!p) return LMOE_ERR_INVALID_ARG;
  if (!aligned16(p)) return LMOE_ERR_INVALID_ARG;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_INVALID_ARG;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Carve {
  size_t off = 0;
  template <typename T>
  size_t take(size_t count) {
    size_t o = off;
    off = align_up(off + count * sizeof(T), 256);
    return o;
  }
};

// Staging buffers, streams and events of lmoe_forward_host (no-op if never created).
void release_host_io(lmoe_ctx* ctx) {
  for (cudaEvent_t* ev : {&ctx->host_in[0], &ctx->host_in[1], &ctx->host_run[0], &ctx->host_run[1],
                          &ctx->host_out[0], &ctx->host_out[1], &ctx->host_last_run, &ctx->host_dev_done}) {
    if (*ev) cudaEventDestroy(*ev);
    *ev = nullptr;
  }
  for (cudaStream_t* st : {&ctx->host_in_st, &ctx->host_run_st, &ctx->host_out_st}) {
    if (*st) cudaStreamDestroy(*st);
    *st = nullptr;
  }
  cudaFree(ctx->host_ws);
  ctx->host_ws = nullptr;
  ctx->host_next = 0;
}

// Device-buffer calls share the context's workspace with the host-buffer forwards, which run on
// the context's own stream: once lmoe_forward_host has been used, a device-buffer call waits for
// the last host-buffer forward and marks where its own work ends (for the next host-buffer one).
void host_order_begin(lmoe_ctx* ctx, cudaStream_t st) {
  if (ctx && ctx->host_ws) cudaStreamWaitEvent(st, ctx->host_last_run, 0);
}

void host_order_end(lmoe_ctx* ctx, cudaStream_t st) {
  if (ctx && ctx->host_ws) cudaEventRecord(ctx->host_dev_done, st);
}

// Synchronise `st`, then read and clear the context's device status word.
lmoe_status read_status(lmoe_ctx* ctx, cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return LMOE_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ctx->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LMOE_ERR_CUDA;
  if (v && cudaMemset(ctx->status, 0, 4) != cudaSuccess) return LMOE_ERR_CUDA;
  if (v & kStatusTimeout) return LMOE_ERR_TIMEOUT;
  if (v & kStatusAssert) return LMOE_ERR_DEVICE_ASSERT;
  return LMOE_OK;
}

lmoe_status finish(lmoe_ctx* ctx, cudaStream_t st, cudaError_t e) {
  if (e != cudaSuccess) return LMOE_ERR_CUDA;
  if (ctx->check) return read_status(ctx, st);
  return LMOE_OK;
}

cudaError_t run_gemm(lmoe_ctx* ctx, const GemmArgs& g, cudaStream_t st) {
  if (ctx->use_tc) {
    int n = 0;
    const cudaError_t e = launch_gemm_tc(ctx->tc, g, st, &n);
    ctx->launches += n;
    return e;
  }
  ctx->launches += 1;
  return launch_gemm_simt(g, ctx->bf16, st);
}

GemmArgs base_args(const lmoe_ctx* ctx) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.nseg = 1;
  g.beta = ctx->cfg.beta;
  g.beta_u = ctx->cfg.beta_u;
  return g;
}

cudaError_t route_impl(lmoe_ctx* ctx, const void* x, int bt, cudaStream_t st, int32_t* user_counts) {
  const lmoe_config& c = ctx->cfg;
  GemmArgs g = base_args(ctx);
  g.M = bt; g.N = c.n_experts; g.K = c.d;
  g.A = x; g.lda = c.d;
  g.seg_k0[0] = 0; g.seg_k0[1] = c.d;
  g.seg_B[0] = ctx->w.w_router; g.seg_ldb[0] = c.d;
  g.epi = kEpiRouter;
  g.out = ctx->logits; g.ldo = c.n_experts;
  g.out_t = ctx->logits_t; g.ldt = bt;
  g.bias = ctx->w.router_bias;
  g.op = kOpRouter;
  cudaError_t e = run_gemm(ctx, g, st);
  if (e != cudaSuccess) return e;
  stage_mark(ctx, 1, st);
  RouteArgs r;
  r.logits = ctx->logits; r.logits_t = ctx->logits_t;
  r.bt = bt; r.n_experts = c.n_experts; r.top_k = c.top_k; r.tile_m = ctx->use_tc ? tc_group_tile(ctx->tc) : kTileM;
  r.alpha = ctx->alpha; r.idx = ctx->idx; r.w = ctx->wk;
  r.block_cnt = ctx->block_cnt; r.counts = ctx->counts; r.offsets = ctx->offsets;
  r.mtile_off = ctx->mtile_off; r.perm = ctx->perm; r.inv = ctx->inv;
  r.user_counts = user_counts;
  r.sm_count = ctx->sm_count;
  r.list = ctx->topk_list;
  r.list_count = ctx->topk_list + ctx->max_bt;
  r.momentum = ctx->momentum;
  r.alpha_prev = (ctx->momentum > 0.0 && ctx->state_valid) ? ctx->alpha_state : nullptr;
  r.alpha_state = ctx->momentum > 0.0 ? ctx->alpha_state : nullptr;
  ctx->launches += kRouteTailLaunches;
  e = launch_route_tail(r, st);
  if (e == cudaSuccess && ctx->momentum > 0.0) ctx->state_valid = true;
  return e;
}

// Runs the segment validation on the index buffers of the last bt tokens routed, then
// synchronises `st` and returns (and clears) the status word.
lmoe_status validate_routing(lmoe_ctx* ctx, int bt, cudaStream_t st) {
  const lmoe_config& c = ctx->cfg;
  ctx->launches += 1;
  if (launch_validate_segments(ctx->idx, ctx->counts, ctx->offsets, ctx->perm, ctx->inv, bt, c.top_k, c.n_experts,
                               ctx->status, ctx->sm_count, st) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  return read_status(ctx, st);
}

}  // namespace

extern "C" {

const char* lmoe_status_string(lmoe_status s) {
  switch (s) {
    case LMOE_OK: return "LMOE_OK";
    case LMOE_ERR_INVALID_ARG: return "LMOE_ERR_INVALID_ARG";
    case LMOE_ERR_UNSUPPORTED: return "LMOE_ERR_UNSUPPORTED";
    case LMOE_ERR_OOM: return "LMOE_ERR_OOM";
    case LMOE_ERR_CUDA: return "LMOE_ERR_CUDA";
    case LMOE_ERR_TIMEOUT: return "LMOE_ERR_TIMEOUT";
    case LMOE_ERR_DEVICE_ASSERT: return "LMOE_ERR_DEVICE_ASSERT";
  }
  return "LMOE_ERR_UNKNOWN";
}

const char* lmoe_build_info(void) {
  return "lmoe sm_103a: bf16 = tcgen05/TMEM/TMA GEMMs, fp32 = CUDA-core fp32 FMA GEMMs";
}

}  // extern "C"

namespace {

// lmoe_create, lmoe_create_fp8 (f8 != nullptr: e4m3 routed experts) and lmoe_create_mxfp4
// (mx != nullptr: MXFP4 routed experts; their tokens and h are e4m3 as with f8).
lmoe_status create_impl(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_fp8_experts* f8,
                        const lmoe_mxfp4_experts* mx, int32_t max_bt, lmoe_stream stream, lmoe_ctx** out) {
  if (!out) return LMOE_ERR_INVALID_ARG;
  *out = nullptr;
  lmoe_status s = check_cfg(cfg);
  if (s != LMOE_OK) return s;
  if (!w) return LMOE_ERR_INVALID_ARG;
  if (max_bt <= 0 || max_bt > (1 << 20)) return LMOE_ERR_INVALID_ARG;
  if ((long long)max_bt * cfg->top_k >= (1LL << 31)) return LMOE_ERR_UNSUPPORTED;
  const bool lowp = f8 || mx;
  if (lowp && cfg->dtype != LMOE_BF16) return LMOE_ERR_INVALID_ARG;
  const void* req[] = {w->w_router, w->w_down, w->latent_gamma, w->w_up, w->sh_gate, w->sh_up, w->sh_down,
                       f8 ? f8->exp_gate : mx ? mx->exp_gate : w->exp_gate,
                       f8 ? f8->exp_up : mx ? mx->exp_up : w->exp_up,
                       f8 ? f8->exp_down : mx ? mx->exp_down : w->exp_down};
  for (const void* p : req)
    if (!p || !aligned16(p)) return LMOE_ERR_INVALID_ARG;
  if (w->router_bias && !aligned16(w->router_bias)) return LMOE_ERR_INVALID_ARG;
  if (f8) {
    const float* sc[] = {f8->gate_scale, f8->up_scale, f8->down_scale};
    for (const float* p : sc)
      if (!p || (reinterpret_cast<uintptr_t>(p) & 3u)) return LMOE_ERR_INVALID_ARG;
  }
  if (mx) {
    // TMA reads the packed codes from 32-byte aligned rows; the scale groups are bulk-copied
    const void* codes[] = {mx->exp_gate, mx->exp_up, mx->exp_down};
    for (const void* p : codes)
      if (reinterpret_cast<uintptr_t>(p) & 31u) return LMOE_ERR_INVALID_ARG;
    const void* sc[] = {mx->gate_sf, mx->up_sf, mx->down_sf};
    for (const void* p : sc)
      if (!p || !aligned16(p)) return LMOE_ERR_INVALID_ARG;
    if (cfg->latent % 128 || cfg->expert_inter % 128) return LMOE_ERR_UNSUPPORTED;
  }
  // from here on the CUDA runtime is needed
  for (const void* p : req)
    if ((s = check_device_ptr(p)) != LMOE_OK) return s;
  if (w->router_bias && (s = check_device_ptr(w->router_bias)) != LMOE_OK) return s;
  if (lowp) {
    const void* sc8[] = {f8 ? (const void*)f8->gate_scale : nullptr, f8 ? (const void*)f8->up_scale : nullptr,
                         f8 ? (const void*)f8->down_scale : nullptr};
    const void* scmx[] = {mx ? mx->gate_sf : nullptr, mx ? mx->up_sf : nullptr, mx ? mx->down_sf : nullptr};
    for (const void* p : (f8 ? sc8 : scmx)) {
      cudaPointerAttributes at;
      if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return LMOE_ERR_INVALID_ARG;
      }
      if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return LMOE_ERR_INVALID_ARG;
    }
  }

  lmoe_ctx* ctx = new (std::nothrow) lmoe_ctx();
  if (!ctx) return LMOE_ERR_OOM;
  ctx->cfg = *cfg;
  ctx->w = *w;
  ctx->max_bt = max_bt;
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->bf16 = cfg->dtype == LMOE_BF16;
  ctx->f8 = lowp;
  ctx->esz = ctx->bf16 ? 2 : 4;
  const char* chk = getenv("LMOE_CHECK");
  ctx->check = chk && chk[0] == '1';
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess ||
      route_tail_prepare() != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return LMOE_ERR_CUDA;
  }

  const lmoe_config& c = *cfg;
  const size_t bt = (size_t)max_bt, E = c.n_experts, K = c.top_k, L = c.latent;
  const size_t nblk = (bt + kSegTokens - 1) / kSegTokens;
  const size_t ldc = L + (size_t)c.n_shared * c.shared_inter;
  Carve cv;
  size_t o_logits = cv.take<float>(bt * E);
  size_t o_logits_t = cv.take<float>(bt * E);
  size_t o_alpha = cv.take<double>(E);
  size_t o_alpha_state = cv.take<double>(E);
  size_t o_idx = cv.take<int32_t>(bt * K);
  size_t o_w = cv.take<float>(bt * K);
  size_t o_bcnt = cv.take<int32_t>(nblk * E);
  size_t o_cnt = cv.take<int32_t>(E);
  size_t o_off = cv.take<int32_t>(E + 1);
  size_t o_mt = cv.take<int32_t>(E + 1);
  size_t o_perm = cv.take<int32_t>(bt * K);
  size_t o_inv = cv.take<int32_t>(bt * K);
  size_t o_list = cv.take<int32_t>(bt + 1);
  size_t o_status = cv.take<uint32_t>(4);
  size_t o_z = cv.take<char>(bt * L * ctx->esz);
  size_t o_zq = lowp ? cv.take<char>(bt * L) : 0;
  size_t o_zp = ctx->bf16 ? cv.take<char>(bt * K * L * 2) : 0;
  size_t o_h = cv.take<char>(bt * K * c.expert_inter * ctx->esz);
  size_t o_y = cv.take<char>(bt * K * L * ctx->esz);
  size_t o_cat = cv.take<char>(bt * ldc * ctx->esz);
  size_t o_tscale = cv.take<float>(bt);
  size_t o_part = ctx->bf16 ? cv.take<float>((size_t)ctx->sm_count * kTcPartPerSm) : 0;
  ctx->ws_bytes = cv.off;
  if (ws_malloc(reinterpret_cast<void**>(&ctx->ws), ctx->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return LMOE_ERR_OOM;
  }
  char* b = ctx->ws;
  ctx->logits = (float*)(b + o_logits);
  ctx->logits_t = (float*)(b + o_logits_t);
  ctx->alpha = (double*)(b + o_alpha);
  ctx->alpha_state = (double*)(b + o_alpha_state);
  ctx->idx = (int32_t*)(b + o_idx);
  ctx->wk = (float*)(b + o_w);
  ctx->block_cnt = (int32_t*)(b + o_bcnt);
  ctx->counts = (int32_t*)(b + o_cnt);
  ctx->offsets = (int32_t*)(b + o_off);
  ctx->mtile_off = (int32_t*)(b + o_mt);
  ctx->perm = (int32_t*)(b + o_perm);
  ctx->inv = (int32_t*)(b + o_inv);
  ctx->topk_list = (int32_t*)(b + o_list);
  ctx->status = (uint32_t*)(b + o_status);
  ctx->z = b + o_z;
  ctx->zq = lowp ? b + o_zq : nullptr;
  ctx->zp = ctx->bf16 ? b + o_zp : nullptr;
  ctx->h = b + o_h;
  ctx->y = b + o_y;
  ctx->cat = b + o_cat;
  ctx->tscale = (float*)(b + o_tscale);
  ctx->part = ctx->bf16 ? (float*)(b + o_part) : nullptr;
  if (cudaMemset(ctx->ws, 0, ctx->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(ctx->ws);
    delete ctx;
    return LMOE_ERR_CUDA;
  }
  ctx->use_tc = false;
  ctx->tc = nullptr;
  if (ctx->bf16) {
    const char* force = getenv("LMOE_FORCE_SIMT");
    if (lowp && force && force[0] == '1') {
      cudaFree(ctx->ws);
      delete ctx;
      return LMOE_ERR_UNSUPPORTED;
    }
    if (!(force && force[0] == '1')) {
      TcBuffers tb;
      tb.z = ctx->z; tb.zq = ctx->zq; tb.zp = ctx->zp; tb.h = ctx->h; tb.y = ctx->y; tb.cat = ctx->cat;
      tb.tscale = ctx->tscale;
      tb.part = ctx->part;
      tb.status = ctx->status;
      lmoe_status ts = tc_plan_create(&c, w, f8, mx, max_bt, ctx->sm_count, tb, &ctx->tc);
      if (ts != LMOE_OK) {
        cudaFree(ctx->ws);
        delete ctx;
        return ts;
      }
      ctx->use_tc = ctx->tc != nullptr;
    }
  }
  *out = ctx;
  return LMOE_OK;
}

}  // namespace

extern "C" {

lmoe_status lmoe_create(const lmoe_config* cfg, const lmoe_weights* w, int32_t max_bt, lmoe_stream stream,
                        lmoe_ctx** out) {
  return logged("lmoe_create", create_impl(cfg, w, nullptr, nullptr, max_bt, stream, out));
}

lmoe_status lmoe_create_fp8(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_fp8_experts* experts,
                            int32_t max_bt, lmoe_stream stream, lmoe_ctx** out) {
  if (!experts) {
    if (out) *out = nullptr;
    return logged("lmoe_create_fp8", LMOE_ERR_INVALID_ARG);
  }
  return logged("lmoe_create_fp8", create_impl(cfg, w, experts, nullptr, max_bt, stream, out));
}

lmoe_status lmoe_create_mxfp4(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_mxfp4_experts* experts,
                              int32_t max_bt, lmoe_stream stream, lmoe_ctx** out) {
  if (!experts) {
    if (out) *out = nullptr;
    return logged("lmoe_create_mxfp4", LMOE_ERR_INVALID_ARG);
  }
  return logged("lmoe_create_mxfp4", create_impl(cfg, w, nullptr, experts, max_bt, stream, out));
}

static lmoe_status route_entry(lmoe_ctx* ctx, const void* x, int32_t bt, lmoe_stream stream,
                               int32_t* topk_idx, float* topk_w, int32_t* expert_counts, double* alpha,
                               float* logits) {
  if (!ctx || bt < 0 || bt > ctx->max_bt) return LMOE_ERR_INVALID_ARG;
  if (bt == 0) return LMOE_OK;
  if (!x || !aligned16(x)) return LMOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const lmoe_config& c = ctx->cfg;
  ctx->last_bt = bt;
  cudaError_t e = route_impl(ctx, x, bt, st, expert_counts);
  if (e == cudaSuccess && ctx->check) {
    const lmoe_status vs = validate_routing(ctx, bt, st);
    if (vs != LMOE_OK) return vs;
  }
  const size_t btK = (size_t)bt * c.top_k;
  if (e == cudaSuccess && topk_idx)
    e = cudaMemcpyAsync(topk_idx, ctx->idx, btK * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && topk_w)
    e = cudaMemcpyAsync(topk_w, ctx->wk, btK * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && alpha)
    e = cudaMemcpyAsync(alpha, ctx->alpha, (size_t)c.n_experts * 8, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && logits)
    e = cudaMemcpyAsync(logits, ctx->logits, (size_t)bt * c.n_experts * 4, cudaMemcpyDeviceToDevice, st);
  return finish(ctx, st, e);
}

static lmoe_status forward_entry(lmoe_ctx* ctx, const void* x, int32_t bt, void* out, lmoe_stream stream) {
  if (!ctx || bt < 0 || bt > ctx->max_bt) return LMOE_ERR_INVALID_ARG;
  if (bt == 0) return LMOE_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return LMOE_ERR_INVALID_ARG;
  const lmoe_config& c = ctx->cfg;
  const size_t xbytes = (size_t)bt * c.d * ctx->esz;
  const char* xb = static_cast<const char*>(x);
  const char* ob = static_cast<const char*>(out);
  if (ob < xb + xbytes && xb < ob + xbytes) return LMOE_ERR_INVALID_ARG;  // out overlaps x
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ctx->last_bt = bt;
  nvtxRangePushA("lmoe_forward");
  ctx->nvtx_open = 1;
  stage_mark(ctx, 0, st);
  cudaError_t e = route_impl(ctx, x, bt, st, nullptr);
  stage_mark(ctx, 2, st);
  if (e == cudaSuccess && ctx->check) {  // check mode: the segments are verified before any kernel indexes through them
    const lmoe_status vs = validate_routing(ctx, bt, st);
    if (vs != LMOE_OK) {
      nvtx_end(ctx);
      return vs;
    }
  }
  const long long ldc = (long long)c.latent + (long long)c.n_shared * c.shared_inter;
  const int tile_m = ctx->use_tc ? tc_group_tile(ctx->tc) : kTileM;
  const int max_mtiles = (int)(((long long)bt * c.top_k) / tile_m + c.n_experts + 1);  // >= sum of ceil(cnt/tile_m)

  if (e == cudaSuccess) {  // z = x W_down^T
    GemmArgs g = base_args(ctx);
    g.M = bt; g.N = c.latent; g.K = c.d;
    g.A = x; g.lda = c.d;
    g.seg_k0[1] = c.d; g.seg_B[0] = ctx->w.w_down; g.seg_ldb[0] = c.d;
    g.epi = kEpiStore; g.out = ctx->z; g.ldo = c.latent;
    g.op = kOpDown;
    e = run_gemm(ctx, g, st);
    stage_mark(ctx, 3, st);
  }
  if (e == cudaSuccess) {  // h[slot] = act(W_g[e] z[perm[slot]], W_u[e] z[perm[slot]])
    GemmArgs g = base_args(ctx);
    g.M = bt * c.top_k; g.N = c.expert_inter; g.K = c.latent;
    g.A = ctx->z; g.lda = c.latent; g.a_rows = ctx->perm;
    g.seg_k0[1] = c.latent; g.seg_B[0] = ctx->w.exp_gate; g.seg_ldb[0] = c.latent;
    g.B_up = ctx->w.exp_up; g.b_group_rows = c.expert_inter;
    g.seg_off = ctx->offsets; g.mtile_off = ctx->mtile_off; g.G = c.n_experts; g.max_mtiles = max_mtiles;
    g.bt_tokens = bt;
    g.epi = kEpiGlu; g.out = ctx->h; g.ldo = c.expert_inter;
    g.op = kOpExpertGateUp;
    if (ctx->use_tc) {  // the experts' token rows into slot order (the CUDA-core engine reads them through perm)
      int n = 0;
      e = tc_gather_tokens(ctx->tc, g, st, &n);
      ctx->launches += n;
    }
    stage_mark(ctx, 4, st);
    if (e == cudaSuccess) e = run_gemm(ctx, g, st);
    stage_mark(ctx, 5, st);
  }
  if (e == cudaSuccess) {  // y[slot] = W_d[e] h[slot]
    GemmArgs g = base_args(ctx);
    g.M = bt * c.top_k; g.N = c.latent; g.K = c.expert_inter;
    g.A = ctx->h; g.lda = c.expert_inter;
    g.seg_k0[1] = c.expert_inter; g.seg_B[0] = ctx->w.exp_down; g.seg_ldb[0] = c.expert_inter;
    g.b_group_rows = c.latent;
    g.seg_off = ctx->offsets; g.mtile_off = ctx->mtile_off; g.G = c.n_experts; g.max_mtiles = max_mtiles;
    g.bt_tokens = bt;
    g.epi = kEpiStore; g.out = ctx->y; g.ldo = c.latent;
    g.op = kOpExpertDown;
    e = run_gemm(ctx, g, st);
    stage_mark(ctx, 6, st);
  }
  if (e == cudaSuccess) {  // c = sum_k w RMSNorm(y_k) -> cat[:, 0:L]
    CombineArgs a;
    a.y = ctx->y; a.inv = ctx->inv; a.w = ctx->wk; a.gamma = ctx->w.latent_gamma;
    a.bt = bt; a.top_k = c.top_k; a.latent = c.latent; a.eps = c.rms_eps;
    a.cat = ctx->cat; a.ldc = ldc;
    a.norm_sum = ctx->norm_sum;
    e = launch_combine(a, ctx->bf16, st);
    ctx->launches += 1;
    stage_mark(ctx, 7, st);
  }
  if (e == cudaSuccess) {  // shared activations -> cat[:, L:]
    GemmArgs g = base_args(ctx);
    g.M = bt; g.N = c.n_shared * c.shared_inter; g.K = c.d;
    g.A = x; g.lda = c.d;
    g.seg_k0[1] = c.d; g.seg_B[0] = ctx->w.sh_gate; g.seg_ldb[0] = c.d;
    g.B_up = ctx->w.sh_up;
    g.epi = kEpiGlu;
    g.out = static_cast<char*>(ctx->cat) + (size_t)c.latent * ctx->esz; g.ldo = ldc;
    g.op = kOpSharedGateUp;
    e = run_gemm(ctx, g, st);
    stage_mark(ctx, 8, st);
  }
  if (e == cudaSuccess) {  // out = [c | h_sh] [W_up | W_d^sh_0 | ...]^T
    GemmArgs g = base_args(ctx);
    g.M = bt; g.N = c.d; g.K = (int)ldc;
    g.A = ctx->cat; g.lda = ldc;
    g.nseg = 1 + c.n_shared;
    g.seg_k0[0] = 0; g.seg_B[0] = ctx->w.w_up; g.seg_ldb[0] = c.latent; g.seg_row0[0] = 0;
    for (int j = 0; j < c.n_shared; ++j) {
      g.seg_k0[1 + j] = c.latent + j * c.shared_inter;
      g.seg_B[1 + j] = ctx->w.sh_down;
      g.seg_ldb[1 + j] = c.shared_inter;
      g.seg_row0[1 + j] = (long long)j * c.d;
    }
    g.seg_k0[g.nseg] = (int)ldc;
    g.epi = kEpiStore; g.out = out; g.ldo = c.d;
    g.op = kOpFinal;
    e = run_gemm(ctx, g, st);
    stage_mark(ctx, 9, st);
  }
  if (ctx->prof_on && ctx->prof_calls < kProfCap) ctx->prof_calls++;
  nvtx_end(ctx);
  return finish(ctx, st, e);
}

lmoe_status lmoe_set_cutoff_momentum(lmoe_ctx* ctx, double momentum) {
  if (!ctx || !(momentum >= 0.0 && momentum < 1.0)) return LMOE_ERR_INVALID_ARG;
  ctx->momentum = momentum;
  ctx->state_valid = false;
  return LMOE_OK;
}

lmoe_status lmoe_set_latent_norm(lmoe_ctx* ctx, lmoe_latent_norm placement) {
  if (!ctx || (placement != LMOE_NORM_PER_EXPERT && placement != LMOE_NORM_COMBINED)) return LMOE_ERR_INVALID_ARG;
  const bool norm_sum = placement == LMOE_NORM_COMBINED;
  if (norm_sum && ctx->cfg.latent > kMaxNormSumLatent) return LMOE_ERR_UNSUPPORTED;
  if (prepare_combine(ctx->cfg.latent, norm_sum) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  ctx->norm_sum = norm_sum;
  return LMOE_OK;
}

lmoe_status lmoe_debug_inject_wait_timeout(lmoe_ctx* ctx) {
  if (!ctx) return LMOE_ERR_INVALID_ARG;
  if (!ctx->use_tc) return LMOE_ERR_UNSUPPORTED;
  tc_inject_wait_timeout(ctx->tc);
  return LMOE_OK;
}

lmoe_status lmoe_profile(lmoe_ctx* ctx, int32_t enable) {
  if (!ctx) return LMOE_ERR_INVALID_ARG;
  if (enable && ctx->prof_ev.empty()) {
    ctx->prof_ev.resize((size_t)kProfCap * (LMOE_NUM_STAGES + 1));
    for (auto& ev : ctx->prof_ev)
      if (cudaEventCreate(&ev) != cudaSuccess) return LMOE_ERR_CUDA;
  }
  if (enable) { ctx->prof_calls = 0; ctx->prof_launch_base = ctx->launches; }
  ctx->prof_on = enable != 0;
  return LMOE_OK;
}

lmoe_status lmoe_profile_read(lmoe_ctx* ctx, float* ms, int32_t* calls, int64_t* launches) {
  if (!ctx) return LMOE_ERR_INVALID_ARG;
  float acc[LMOE_NUM_STAGES] = {0};
  for (int c = 0; c < ctx->prof_calls; ++c) {
    cudaEvent_t* ev = &ctx->prof_ev[(size_t)c * (LMOE_NUM_STAGES + 1)];
    if (cudaEventSynchronize(ev[LMOE_NUM_STAGES]) != cudaSuccess) return LMOE_ERR_CUDA;
    for (int s = 0; s < LMOE_NUM_STAGES; ++s) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ev[s], ev[s + 1]) != cudaSuccess) return LMOE_ERR_CUDA;
      acc[s] += t;
    }
  }
  if (ms) for (int s = 0; s < LMOE_NUM_STAGES; ++s) ms[s] = acc[s];
  if (calls) *calls = ctx->prof_calls;
  if (launches) *launches = ctx->launches - ctx->prof_launch_base;
  return LMOE_OK;
}

static lmoe_status sync_status_entry(lmoe_ctx* ctx, lmoe_stream stream) {
  if (!ctx) return LMOE_ERR_INVALID_ARG;
  return read_status(ctx, static_cast<cudaStream_t>(stream));
}

static lmoe_status forward_host_entry(lmoe_ctx* ctx, const void* x_host, int32_t bt, void* out_host,
                                      lmoe_stream stream) {
  if (!ctx || bt < 0 || bt > ctx->max_bt) return LMOE_ERR_INVALID_ARG;
  if (bt == 0) return LMOE_OK;
  if (!x_host || !out_host) return LMOE_ERR_INVALID_ARG;
  const size_t bytes = (size_t)bt * ctx->cfg.d * ctx->esz;
  const char* xb = static_cast<const char*>(x_host);
  const char* ob = static_cast<const char*>(out_host);
  if (ob < xb + bytes && xb < ob + bytes) return LMOE_ERR_INVALID_ARG;  // out overlaps x
  for (const void* p : {x_host, static_cast<const void*>(out_host)}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return LMOE_ERR_INVALID_ARG;
    }
    if (at.type != cudaMemoryTypeHost && at.type != cudaMemoryTypeUnregistered) return LMOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t one = align_up((size_t)ctx->max_bt * ctx->cfg.d * ctx->esz, 256);
  if (!ctx->host_ws) {  // first call: staging buffers, streams, events
    if (ws_malloc(reinterpret_cast<void**>(&ctx->host_ws), 4 * one) != cudaSuccess) {
      cudaGetLastError();
      ctx->host_ws = nullptr;
      return LMOE_ERR_OOM;
    }
    bool ok = true;
    for (cudaStream_t* s2 : {&ctx->host_in_st, &ctx->host_run_st, &ctx->host_out_st})
      ok = ok && cudaStreamCreateWithFlags(s2, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* ev : {&ctx->host_in[0], &ctx->host_in[1], &ctx->host_run[0], &ctx->host_run[1],
                            &ctx->host_out[0], &ctx->host_out[1], &ctx->host_last_run, &ctx->host_dev_done})
      ok = ok && cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess;
    // the device-buffer calls made so far were on the caller's stream
    ok = ok && cudaEventRecord(ctx->host_dev_done, st) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      release_host_io(ctx);
      return LMOE_ERR_CUDA;
    }
  }
  const int b = ctx->host_next;
  char* xd = ctx->host_ws + (size_t)b * one;
  char* od = ctx->host_ws + (size_t)(2 + b) * one;
  // input copy once the forward that last read x[b] is done; it overlaps the previous forward
  cudaError_t e = cudaStreamWaitEvent(ctx->host_in_st, ctx->host_run[b], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, ctx->host_in_st);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->host_in[b], ctx->host_in_st);
  // forward once its input is in, the output copy that last read out[b] is done, and the last
  // device-buffer call on this context is done
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->host_run_st, ctx->host_in[b], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->host_run_st, ctx->host_out[b], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->host_run_st, ctx->host_dev_done, 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  ctx->host_next = b ^ 1;
  const lmoe_status s = forward_entry(ctx, xd, bt, od, ctx->host_run_st);
  if (s != LMOE_OK) return s;
  e = cudaEventRecord(ctx->host_run[b], ctx->host_run_st);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->host_last_run, ctx->host_run_st);
  // output copy on its own stream (it overlaps the next forward); the caller's stream waits for it
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->host_out_st, ctx->host_run[b], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, ctx->host_out_st);
  if (e == cudaSuccess) e = cudaEventRecord(ctx->host_out[b], ctx->host_out_st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ctx->host_out[b], 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  return LMOE_OK;
}

void lmoe_destroy(lmoe_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  release_host_io(ctx);
  for (auto& ev : ctx->prof_ev) cudaEventDestroy(ev);
  tc_plan_destroy(ctx->tc);
  cudaFree(ctx->ws);
  delete ctx;
}

lmoe_status lmoe_route(lmoe_ctx* ctx, const void* x, int32_t bt, lmoe_stream stream, int32_t* topk_idx,
                       float* topk_w, int32_t* expert_counts, double* alpha, float* logits) {
  nvtxRangePushA("lmoe_route");
  host_order_begin(ctx, static_cast<cudaStream_t>(stream));
  const lmoe_status s = route_entry(ctx, x, bt, stream, topk_idx, topk_w, expert_counts, alpha, logits);
  host_order_end(ctx, static_cast<cudaStream_t>(stream));
  nvtxRangePop();
  return logged("lmoe_route", s);
}

lmoe_status lmoe_forward(lmoe_ctx* ctx, const void* x, int32_t bt, void* out, lmoe_stream stream) {
  host_order_begin(ctx, static_cast<cudaStream_t>(stream));
  const lmoe_status s = forward_entry(ctx, x, bt, out, stream);
  host_order_end(ctx, static_cast<cudaStream_t>(stream));
  return logged("lmoe_forward", s);
}

lmoe_status lmoe_forward_host(lmoe_ctx* ctx, const void* x_host, int32_t bt, void* out_host, lmoe_stream stream) {
  return logged("lmoe_forward_host", forward_host_entry(ctx, x_host, bt, out_host, stream));
}

lmoe_status lmoe_sync_status(lmoe_ctx* ctx, lmoe_stream stream) {
  return logged("lmoe_sync_status", sync_status_entry(ctx, stream));
}

lmoe_status lmoe_debug_check_segments(lmoe_ctx* ctx, lmoe_stream stream) {
  if (!ctx) return logged("lmoe_debug_check_segments", LMOE_ERR_INVALID_ARG);
  if (ctx->last_bt == 0) return LMOE_OK;
  host_order_begin(ctx, static_cast<cudaStream_t>(stream));
  return logged("lmoe_debug_check_segments", validate_routing(ctx, ctx->last_bt, static_cast<cudaStream_t>(stream)));
}

void lmoe_debug_fail_next_alloc(void) { g_fail_next_alloc.store(1); }

lmoe_status lmoe_workspace(const lmoe_ctx* ctx, lmoe_workspace_view* v) {
  if (!ctx || !v) return LMOE_ERR_INVALID_ARG;
  v->bt = ctx->last_bt;
  v->logits = ctx->logits;
  v->alpha = ctx->alpha;
  v->topk_idx = ctx->idx;
  v->topk_w = ctx->wk;
  v->offsets = ctx->offsets;
  v->perm = ctx->perm;
  v->inv = ctx->inv;
  v->z = ctx->z;
  v->h = ctx->h;
  v->y = ctx->y;
  v->cat = ctx->cat;
  return LMOE_OK;
}

}  // extern "C"
