// C ABI of the dense SiTU-GLU FFN: the full-width feed-forward block of the model's first
// (dense) layer ("Vue d'ensemble de l'architecture", table "Le budget de paramètres, module
// par module": one dense FFN of 727 M parameters, intermediate 33 792 at d = 7168), with the
// SiTU-GLU activation of the experts ("KimiK3的StableLatentMoE架构解析", ¶"第一").
//   out = W_down act(W_gate x, W_up x),  act(g, u) = g' sigmoid(g') u'.
// It runs on the tensor-core GEMM engine of the layer: one SiTU-GLU launch and one store
// launch per call.
#include <cstring>
#include <new>

#include "../../include/lmoe.h"
#include "common.cuh"
#include "gemm_tc.h"

using namespace lmoe;

struct lmoe_ffn {
  lmoe_ffn_config cfg;
  int max_bt;
  int sm_count;
  void* h;               // [max_bt, inter] bf16 activations
  uint32_t* status;      // device status word
  void* ws;              // one allocation: status word, then h
  TcFfnPlan* tc;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lmoe_status check_weight(const void* p) {
  if (!p || !aligned16(p)) return LMOE_ERR_INVALID_ARG;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_INVALID_ARG;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

}  // namespace

extern "C" {

lmoe_status lmoe_ffn_create(const lmoe_ffn_config* cfg, const void* w_gate, const void* w_up, const void* w_down,
                            int32_t max_bt, lmoe_ffn** out) {
  if (!out) return LMOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || cfg->d <= 0 || cfg->inter <= 0 || !(cfg->beta > 0.f) || !(cfg->beta_u > 0.f) ||
      cfg->beta > 3.0e38f || cfg->beta_u > 3.0e38f)
    return LMOE_ERR_INVALID_ARG;
  if (max_bt <= 0 || max_bt > (1 << 20)) return LMOE_ERR_INVALID_ARG;
  if (cfg->d % 64 || cfg->inter % 64) return LMOE_ERR_UNSUPPORTED;
  if ((long long)cfg->inter * cfg->d >= (1LL << 40)) return LMOE_ERR_UNSUPPORTED;
  lmoe_status s;
  if ((s = check_weight(w_gate)) != LMOE_OK || (s = check_weight(w_up)) != LMOE_OK ||
      (s = check_weight(w_down)) != LMOE_OK)
    return s;
  lmoe_ffn* f = new (std::nothrow) lmoe_ffn();
  if (!f) return LMOE_ERR_OOM;
  f->cfg = *cfg;
  f->max_bt = max_bt;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&f->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    delete f;
    return LMOE_ERR_CUDA;
  }
  const size_t h_bytes = (size_t)max_bt * cfg->inter * 2;
  if (cudaMalloc(&f->ws, 256 + h_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete f;
    return LMOE_ERR_OOM;
  }
  f->status = static_cast<uint32_t*>(f->ws);
  f->h = static_cast<char*>(f->ws) + 256;
  if (cudaMemset(f->ws, 0, 256) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(f->ws);
    delete f;
    return LMOE_ERR_CUDA;
  }
  s = tc_ffn_create(cfg->d, cfg->inter, cfg->beta, cfg->beta_u, w_gate, w_up, w_down, max_bt, f->sm_count, f->h,
                    f->status, &f->tc);
  if (s != LMOE_OK) {
    cudaFree(f->ws);
    delete f;
    return s;
  }
  *out = f;
  return LMOE_OK;
}

lmoe_status lmoe_ffn_forward(lmoe_ffn* f, const void* x, int32_t bt, void* out, lmoe_stream stream) {
  if (!f || bt < 0 || bt > f->max_bt) return LMOE_ERR_INVALID_ARG;
  if (bt == 0) return LMOE_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out)) return LMOE_ERR_INVALID_ARG;
  const size_t xbytes = (size_t)bt * f->cfg.d * 2;
  const char* xb = static_cast<const char*>(x);
  const char* ob = static_cast<const char*>(out);
  if (ob < xb + xbytes && xb < ob + xbytes) return LMOE_ERR_INVALID_ARG;  // out overlaps x
  const cudaError_t e = tc_ffn_forward(f->tc, x, bt, out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

lmoe_status lmoe_ffn_sync_status(lmoe_ffn* f, lmoe_stream stream) {
  if (!f) return LMOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LMOE_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, f->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return LMOE_ERR_CUDA;
  if (v && cudaMemset(f->status, 0, 4) != cudaSuccess) return LMOE_ERR_CUDA;
  if (v & kStatusTimeout) return LMOE_ERR_TIMEOUT;
  if (v & kStatusAssert) return LMOE_ERR_DEVICE_ASSERT;
  return LMOE_OK;
}

void lmoe_ffn_destroy(lmoe_ffn* f) {
  if (!f) return;
  cudaDeviceSynchronize();
  tc_ffn_destroy(f->tc);
  cudaFree(f->ws);
  delete f;
}

}  // extern "C"
