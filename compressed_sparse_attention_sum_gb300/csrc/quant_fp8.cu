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

// eight values times inv -> eight e4m3 codes at p (8-byte aligned)
__device__ __forceinline__ void store_codes8(uint8_t* p, const float (&v)[8], float inv) {
  uint2 u;
  u.x = (uint32_t)e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
        ((uint32_t)e4m3x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 16);
  u.y = (uint32_t)e4m3x2(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv)) |
        ((uint32_t)e4m3x2(__fmul_rn(v[6], inv), __fmul_rn(v[7], inv)) << 16);
  *reinterpret_cast<uint2*>(p) = u;
}

// Eight elements held in their storage format (16 bytes of bf16, 32 of fp32)
// so that R rows in flight cost few registers.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    u = __ldg(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);            // bf16 -> fp32 is exact
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p + 4));
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

// G lanes per row (G a power of two, 8 G <= d), R rows per lane group: the
// first 8-element chunk of each of the R rows is loaded before any reduction
// so that R loads are in flight per thread; chunks beyond the first G per
// row (d > 8 G) are re-read in the second pass.
template <typename T, int G, int R>
__global__ void __launch_bounds__(256, 4) quantize_e4m3_kernel(const T* __restrict__ x,
                                                               long long rows, int d,
                                                               uint8_t* __restrict__ out,
                                                               float* __restrict__ scale) {
  constexpr int kRowsPerPass = 32 / G;
  const int lane = threadIdx.x & 31, lg = lane % G;
  const long long warp_id = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const long long row0 = warp_id * (R * kRowsPerPass) + lane / G;
  const int nchunk = d / 8;
  Raw8<T> raw[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const long long row = row0 + (long long)r * kRowsPerPass;
    if (row < rows) raw[r].load(x + row * d + lg * 8);
    else raw[r].zero();
  }
  float amax[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const long long row = row0 + (long long)r * kRowsPerPass;
    float v[8];
    raw[r].get(v);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
    if (row < rows) {
      for (int ch = lg + G; ch < nchunk; ch += G) {
        float u[8];
        load8(x + row * d + ch * 8, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(u[e]));
      }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    amax[r] = m;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const long long row = row0 + (long long)r * kRowsPerPass;
    if (row >= rows) continue;
    const float inv = amax[r] > 0.f ? __fdiv_rn(448.f, amax[r]) : 0.f;
    if (lg == 0) scale[row] = __fdiv_rn(amax[r], 448.f);
    uint8_t* orow = out + row * d;
    float v[8];
    raw[r].get(v);
    store_codes8(orow + lg * 8, v, inv);
    for (int ch = lg + G; ch < nchunk; ch += G) {
      float u[8];
      load8(x + row * d + ch * 8, u);
      store_codes8(orow + ch * 8, u, inv);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void* x, long long rows, int d, bool bf16, uint8_t* out,
                                 float* scale, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  constexpr int R = 4;
  const int chunks = d / 8;
  const int G = chunks >= 32 ? 32 : chunks >= 16 ? 16 : chunks >= 8 ? 8 : chunks >= 4 ? 4
              : chunks >= 2 ? 2 : 1;
  const long long rows_per_cta = 8ll * R * (32 / G);
  const unsigned grid = (unsigned)((rows + rows_per_cta - 1) / rows_per_cta);
#define CSA_QUANT(GG)                                                                            \
  if (G == GG) {                                                                                 \
    if (bf16)                                                                                    \
      quantize_e4m3_kernel<__nv_bfloat16, GG, R><<<grid, 256, 0, s>>>(                           \
          (const __nv_bfloat16*)x, rows, d, out, scale);                                         \
    else                                                                                         \
      quantize_e4m3_kernel<float, GG, R><<<grid, 256, 0, s>>>((const float*)x, rows, d, out,     \
                                                              scale);                            \
  }
  CSA_QUANT(32) CSA_QUANT(16) CSA_QUANT(8) CSA_QUANT(4) CSA_QUANT(2) CSA_QUANT(1)
#undef CSA_QUANT
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
