// Tensor-core (tcgen05 / TMEM / TMA) GEMM engine of the bf16 layer.
#pragma once

#include "../../include/lmoe.h"
#include "internal.h"

namespace lmoe {

struct TcPlan;  // tensor maps of the borrowed weights and of the workspace, launch shapes

struct TcBuffers {
  void* z;           // [max_bt, latent] bf16: the routed experts gather their token rows from it
  void* zq;          // [max_bt, latent] e4m3 copy of z (fp8 experts only)
  void* zp;          // [max_bt * K, latent] routed token rows in slot order (bf16, or e4m3 bytes)
  void* h;
  void* y;
  void* cat;
  float* tscale;     // [max_bt] per-token scales of zq (fp8 experts)
  float* part;       // [sm_count * 65536] fp32 split-K partial accumulators of the dense GEMMs
  uint32_t* status;
};

// Builds the weight / workspace descriptors.  *plan == nullptr with LMOE_OK means the
// engine does not cover this configuration.
// f8 != nullptr: routed experts in e4m3 (w's expert pointers are not used); h then holds
// e4m3 bytes.
// mx != nullptr: routed experts in MXFP4 (e2m1 codes with tiled ue8m0 block scales), with e4m3
// token rows and h as for f8.
lmoe_status tc_plan_create(const lmoe_config* cfg, const lmoe_weights* w, const lmoe_fp8_experts* f8,
                           const lmoe_mxfp4_experts* mx, int max_bt, int sm_count, const TcBuffers& buf, TcPlan** plan);
void tc_plan_destroy(TcPlan* plan);
// Test hook: the next routed-expert gate/up launch leaves its token stages unfilled and
// shortens its waits to 20 ms, so the kernel times out, records LMOE timeout status and
// returns.
void tc_inject_wait_timeout(TcPlan* plan);
// Tokens per tile of the routed-expert GEMMs: the granularity of the m-tile prefix the routing
// tail must write for this plan (kTileWide for bf16 / e4m3 experts, kTileM for MXFP4).
int tc_group_tile(const TcPlan* plan);
// One GemmOp; *n = kernels launched (a dense GEMM split along K adds its reduction).
cudaError_t launch_gemm_tc(TcPlan* plan, const GemmArgs& a, cudaStream_t st, int* n);
// fp32 values of TcBuffers::part per SM
constexpr long long kTcPartPerSm = 65536;
// The routed experts' token rows in slot order for the next expert gate/up GEMM (a = its
// GemmArgs): z rows gathered through the slot -> token map, or, with e4m3 experts, z
// quantized once per token and its e4m3 rows gathered.  Returns the kernels launched in *n.
cudaError_t tc_gather_tokens(TcPlan* plan, const GemmArgs& a, cudaStream_t st, int* n);

// Dense SiTU-GLU FFN (out = W_down act(W_gate x, W_up x)) on the same engine: descriptors of
// the borrowed weights and of the caller-provided h [max_bt, inter] buffer.
struct TcFfnPlan;
lmoe_status tc_ffn_create(int d, int inter, float beta, float beta_u, const void* w_gate, const void* w_up,
                          const void* w_down, int max_bt, int sm_count, void* h, uint32_t* status, TcFfnPlan** plan);
void tc_ffn_destroy(TcFfnPlan* plan);
cudaError_t tc_ffn_forward(TcFfnPlan* plan, const void* x, int bt, void* out, cudaStream_t st);
constexpr int kFfnLaunches = 2;

}  // namespace lmoe
