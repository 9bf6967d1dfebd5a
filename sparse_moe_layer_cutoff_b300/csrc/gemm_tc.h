// Tensor-core (tcgen05 / TMEM / TMA) GEMM engine of the bf16 layer.
#pragma once

#include "../../include/lmoe.h"
#include "internal.h"

namespace lmoe {

struct TcPlan;  // tensor maps of the borrowed weights and of the workspace, launch shapes

struct TcBuffers {
  void* z;
  void* zp;          // [max_bt * K, latent] routed token rows in slot order
  void* h;
  void* y;
  void* cat;
  uint32_t* status;
};

// Builds the weight / workspace descriptors.  *plan == nullptr with LMOE_OK means the
// engine does not cover this configuration.
lmoe_status tc_plan_create(const lmoe_config* cfg, const lmoe_weights* w, int max_bt, int sm_count,
                           const TcBuffers& buf, TcPlan** plan);
void tc_plan_destroy(TcPlan* plan);
cudaError_t launch_gemm_tc(TcPlan* plan, const GemmArgs& a, cudaStream_t st);
int tc_launches(int op);   // kernels launch_gemm_tc starts for one GemmOp

}  // namespace lmoe
