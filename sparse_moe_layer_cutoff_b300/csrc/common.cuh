// Device helpers shared by the Stable LatentMoE kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lmoe {

typedef __nv_bfloat16 bf16;

// Device status word bits (set with atomicOr, read by lmoe_sync_status).
enum : uint32_t {
  kStatusTimeout = 1u,   // a bounded wait ran out; the kernel returned early
  kStatusAssert = 2u,    // an internal consistency check failed
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// Logistic function in fp64 (router scores are compared in fp64).
__device__ __forceinline__ double sigmoid_f64(double v) { return 1.0 / (1.0 + exp(-v)); }

// SiTU-GLU in fp32: g' = beta tanh(g / beta), u' = beta_u tanh(u / beta_u), act = g' sigmoid(g') u'.
__device__ __forceinline__ float situ_glu(float g, float u, float beta, float beta_u) {
  float gp = beta * tanhf(g / beta);
  float up = beta_u * tanhf(u / beta_u);
  return gp / (1.0f + expf(-gp)) * up;
}

// Order-preserving map between fp32 and uint32 (larger float -> larger key; -0 < +0).
__device__ __forceinline__ uint32_t f32_to_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_f32(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace lmoe
