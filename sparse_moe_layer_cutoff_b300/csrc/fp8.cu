// fp8 (e4m3) routed experts: row quantization of expert weights (an entry point of the
// library) and of the experts' token rows.
//
// "KimiK3的StableLatentMoE架构解析", ¶"第一": the bounded SiTU-GLU output makes fp8 inference
// possible.  Quantization used here, per row of R values:
//   s = absmax / 448 in fp32 (1 for an all-zero row), inv = 1 / s (fp32), q = e4m3(x * inv)
// with e4m3 rounding to nearest, ties to even, saturating at +-448; the row is read back as
// q * s.  Expert weights are quantized once per output row; the experts' input z once per
// token (the expert GEMM gathers the quantized rows of its tokens).
#include <cuda_fp8.h>

#include "../../include/lmoe.h"
#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3) << 8) |
         ((uint32_t)__nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3) << 16) |
         ((uint32_t)__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3) << 24);
}

// One warp quantizes one row of `cols` bf16 values (cols a multiple of 8, 16-byte rows).
__device__ __forceinline__ void quantize_row_warp(const bf16* __restrict__ src, int cols, uint8_t* __restrict__ dst,
                                                  float* __restrict__ scale_out) {
  const int lane = threadIdx.x & 31;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  const int nv = cols / 8;
  float amax = 0.f;
  for (int v = lane; v < nv; v += 32) {
    const uint4 raw = s4[v];
    const bf16* h = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(__bfloat162float(h[i])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
  const float inv = __fdiv_rn(1.0f, s);
  uint2* d2 = reinterpret_cast<uint2*>(dst);
  for (int v = lane; v < nv; v += 32) {
    const uint4 raw = s4[v];
    const bf16* h = reinterpret_cast<const bf16*>(&raw);
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(__bfloat162float(h[i]), inv);
    d2[v] = make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
  }
  if (lane == 0) *scale_out = s;
}

__global__ void __launch_bounds__(256) quantize_rows_kernel(const bf16* __restrict__ w, long long rows, int cols,
                                                            uint8_t* __restrict__ q, float* __restrict__ scale) {
  const long long wpb = blockDim.x >> 5;
  for (long long r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += (long long)gridDim.x * wpb)
    quantize_row_warp(w + r * cols, cols, q + r * cols, scale + r);
}

}  // namespace

cudaError_t launch_quantize_rows(const void* x, long long rows, int cols, void* q, float* scale, int grid,
                                 cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  if (blocks < grid) grid = (int)blocks;
  quantize_rows_kernel<<<grid, 256, 0, st>>>(static_cast<const bf16*>(x), rows, cols, static_cast<uint8_t*>(q), scale);
  return cudaGetLastError();
}

}  // namespace lmoe

extern "C" lmoe_status lmoe_quantize_fp8_rows(const void* w, int64_t rows, int32_t cols, void* q, float* scale,
                                              lmoe_stream stream) {
  if (rows < 0 || cols <= 0) return LMOE_ERR_INVALID_ARG;
  if (rows == 0) return LMOE_OK;
  if (!w || !q || !scale) return LMOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(q) & 7u) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return LMOE_ERR_INVALID_ARG;
  if (cols % 8) return LMOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  const long long blocks = (rows + 7) / 8, cap = (long long)sms * 64;   // 64 blocks per SM at most
  const int grid = (int)(blocks < cap ? blocks : cap);
  lmoe::quantize_rows_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const lmoe::bf16*>(w), rows, cols, static_cast<uint8_t*>(q), scale);
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}
