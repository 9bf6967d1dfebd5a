// MXFP4 routed-expert weights: the quantizer entry point of the library.
//
// "Sparse by design" (the released model's weights in MXFP4) read with the microscaling FP4
// format of the OCP MX specification: a row is cut into blocks of 32 consecutive values along
// its input (K) axis; a block shares one power-of-two scale X = 2^x, x = floor(log2(amax)) - 2
// clamped to [-127, 127] (-127 for an all-zero block), stored as the unsigned byte x + 127
// (ue8m0); each element is e2m1(w / X), rounded to nearest (ties to even) and saturating at +-6.
//
// Layouts written here are the ones the tensor-core kernel reads directly:
//   * q: e2m1 codes packed two per byte along the row, element 2j in the low nibble of byte j
//     (a TMA map of type 16U4_ALIGN16B expands each 8-byte group to a 16-byte shared-memory chunk,
//     the operand layout of tcgen05.mma kind::mxf8f6f4 for 4-bit values);
//   * sf: for each 128-row block rb and 128-column block kq, 512 bytes at
//     (rb * (cols / 128) + kq) * 512 holding the scale of row r (r % 128 = 32 i + l) and 32-column
//     block j (0..3) of that 128-column block at byte 16 l + 4 i + j: one tcgen05.cp of shape
//     32x128b.warpx4 puts the 4 scales of row r into TMEM column i of the block's 4 columns, lane l
//     of every lane quadrant, byte j (the scale-factor id of the j-th K = 32 step).
#include <cuda_fp4.h>

#include "../../include/lmoe.h"
#include "common.cuh"
#include "internal.h"

namespace lmoe {
namespace {

// Byte offset of the scale of (row r, 32-column block b) in the tiled layout above.
__device__ __forceinline__ long long mx_sf_offset(long long r, int b, int kq_per_row) {
  const long long rb = r >> 7;
  const int rr = (int)(r & 127);
  return (rb * kq_per_row + (b >> 2)) * 512 + 16 * (rr & 31) + 4 * (rr >> 5) + (b & 3);
}

// One thread quantizes one block of 32 bf16 values (64 bytes in, 16 bytes of codes and one
// scale byte out).
__global__ void __launch_bounds__(256) quantize_mxfp4_kernel(const bf16* __restrict__ w, long long rows, int cols,
                                                             uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const int nb = cols / 32;
  const long long total = rows * nb;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / nb;
    const int b = (int)(i - r * nb);
    const uint4* src = reinterpret_cast<const uint4*>(w + r * cols + 32 * b);
    float v[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 raw = src[k];
      const bf16* h = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[8 * k + e] = __bfloat162float(h[e]);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
    // floor(log2 amax) from the exponent field; zero and fp32 subnormals clamp to -127
    const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
    int x = ef == 0 ? -127 : ef - 127 - 2;
    if (x < -127) x = -127;
    const float inv = __uint_as_float((uint32_t)(127 - x) << 23);   // 2^-x, exact
    uint32_t packed[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t code = (uint32_t)__nv_cvt_float_to_fp4(v[8 * k + e] * inv, __NV_E2M1, cudaRoundNearest) & 0xFu;
        word |= code << (4 * e);
      }
      packed[k] = word;
    }
    *reinterpret_cast<uint4*>(q + r * (cols / 2) + 16 * b) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    sf[mx_sf_offset(r, b, cols / 128)] = (uint8_t)(x + 127);
  }
}

}  // namespace
}  // namespace lmoe

extern "C" lmoe_status lmoe_quantize_mxfp4_rows(const void* w, int64_t rows, int32_t cols, void* q, void* sf,
                                                lmoe_stream stream) {
  if (rows < 0 || cols <= 0) return LMOE_ERR_INVALID_ARG;
  if (rows == 0) return LMOE_OK;
  if (!w || !q || !sf) return LMOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u)) return LMOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return LMOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return LMOE_ERR_CUDA;
  }
  const long long total = rows * (cols / 32);
  const long long blocks = (total + 255) / 256, cap = (long long)sms * 16;
  const int grid = (int)(blocks < cap ? blocks : cap);
  lmoe::quantize_mxfp4_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const lmoe::bf16*>(w), rows, cols, static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf));
  return cudaGetLastError() == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}
