// csa_quantize_e4m3: per-row e4m3 quantization for the FP8 indexer.
//
// Row r of x [rows, d] (bf16 or fp32) gets the scale absmax / 448 and the
// codes e4m3(x * (448 / absmax)), rounded to nearest even and saturated at
// the largest finite value 448 (an all-zero row gets scale 0 and zero codes).
// The pages list indexer quantization as not included ("Refactor Deepseek v4
// to use Attention Gym's Compressed Sparse Attention", model description);
// this per-row rule is the repository's reading.  Both the reciprocal and
// the product are plain fp32 operations, so an fp32 reference reproduces the
// rounded values bit for bit.
#include <cuda_bf16.h>
#include <cstdint>

#include "csa_common.cuh"

namespace csa {
namespace {

// two fp32 values -> two e4m3 codes, `lo` in the low byte
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// one warp per row; d a multiple of 8
template <typename T>
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const T* __restrict__ x, long long rows,
                                                            int d, uint8_t* __restrict__ out,
                                                            float* __restrict__ scale) {
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* xr = x + row * d;
  float amax = 0.f;
  for (int c = lane * 8; c < d; c += 256) {
    float v[8];
    load8(xr + c, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
  }
  amax = warp_max(amax);
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  if (lane == 0) scale[row] = __fdiv_rn(amax, 448.f);
  uint8_t* orow = out + row * d;
  for (int c = lane * 8; c < d; c += 256) {
    float v[8];
    load8(xr + c, v);
    uint2 u;
    u.x = (uint32_t)e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
          ((uint32_t)e4m3x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 16);
    u.y = (uint32_t)e4m3x2(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv)) |
          ((uint32_t)e4m3x2(__fmul_rn(v[6], inv), __fmul_rn(v[7], inv)) << 16);
    *reinterpret_cast<uint2*>(orow + c) = u;
  }
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void* x, long long rows, int d, bool bf16, uint8_t* out,
                                 float* scale, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (bf16)
    quantize_e4m3_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, rows, d,
                                                             out, scale);
  else
    quantize_e4m3_kernel<float><<<grid, 256, 0, s>>>((const float*)x, rows, d, out, scale);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
