// csa_compress / csa_compress_bwd: softmax-weighted pooling of `ratio`
// consecutive KV tokens, and its gradient.
//
// "Add unfused SBHD compressed sparse attention" (Megatron-LM PR #6400),
// compressor review: the softmax over the block's tokens, the products and
// the sum stay in fp32 and the pooled row is cast once to the storage dtype.
//
// HBM-bound: each kv and score element is read once and each pooled element
// written once.  One thread owns 8 consecutive channels of one block and
// walks the block's tokens with an online (running max) softmax, so the
// scores are read in a single pass.
#include "csa_common.cuh"
#include "csa_kernels.h"

namespace csa {

template <typename T>
__global__ void __launch_bounds__(128) compress_kernel(const T* __restrict__ kv, long long kv_bs,
                                                       const T* __restrict__ score,
                                                       int score_width, T* __restrict__ out,
                                                       long long out_bs, int sq, int d,
                                                       int ratio, int n_c) {
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int bi = blockIdx.y;
  if (gid >= (long long)n_c * groups) return;
  const int j = (int)(gid / groups);
  const int c0 = (int)(gid % groups) * 8;
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  float m[8], l[8], acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) { m[i] = -INFINITY; l[i] = 0.f; acc[i] = 0.f; }
  for (int t = 0; t < ratio; ++t) {
    float v[8], s[8];
    load8(kvp + (long long)t * d, v);
    if (score_width == 1) {
      const float s1 = to_f(scp[(long long)t]);
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i] = s1;
    } else {
      load8(scp + (long long)t * score_width + c0, s);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float mn = fmaxf(m[i], s[i]);
      const float alpha = expf(m[i] - mn);  // 0 on the first token (m = -inf)
      const float e = expf(s[i] - mn);
      l[i] = l[i] * alpha + e;
      acc[i] = acc[i] * alpha + e * v[i];
      m[i] = mn;
    }
  }
  float r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = acc[i] / l[i];
  store8(out + bi * out_bs + (long long)j * d + c0, r);
}

// Backward of the pooling.  With w_t the softmax weights of a block and
// channel, pooled = sum_t w_t kv_t and g = dL/dpooled:
//   dkv_t    += w_t g                      (accumulated: the raw rows also get
//                                           the attention's gradient)
//   dscore_t  = w_t g (kv_t - pooled)      (per channel; summed over channels
//                                           when one score drives all channels)
// Tokens past the last complete block get no kv gradient and zero dscore.
template <typename T>
__global__ void __launch_bounds__(128) compress_bwd_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ g, long long g_bs, float* __restrict__ dkv, long long dkv_bs,
    float* __restrict__ dscore, int sq, int d, int ratio, int n_c) {
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int bi = blockIdx.y;
  if (gid >= (long long)n_c * groups) return;
  const int j = (int)(gid / groups);
  const int c0 = (int)(gid % groups) * 8;
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  float gv[8];
  load8(g + bi * g_bs + (long long)j * d + c0, gv);
  // softmax statistics of the block (per channel)
  float m[8], l[8], pooled[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) { m[i] = -INFINITY; l[i] = 0.f; pooled[i] = 0.f; }
  for (int t = 0; t < ratio; ++t) {
    float v[8], sc[8];
    load8(kvp + (long long)t * d, v);
    if (score_width == 1) {
      const float s1 = to_f(scp[(long long)t]);
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i] = s1;
    } else {
      load8(scp + (long long)t * score_width + c0, sc);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float mn = fmaxf(m[i], sc[i]);
      const float alpha = expf(m[i] - mn);
      const float e = expf(sc[i] - mn);
      l[i] = l[i] * alpha + e;
      pooled[i] = pooled[i] * alpha + e * v[i];
      m[i] = mn;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) pooled[i] /= l[i];
  for (int t = 0; t < ratio; ++t) {
    float v[8], sc[8], dk[8];
    const long long tok = (long long)j * ratio + t;
    load8(kvp + (long long)t * d, v);
    if (score_width == 1) {
      const float s1 = to_f(scp[(long long)t]);
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i] = s1;
    } else {
      load8(scp + (long long)t * score_width + c0, sc);
    }
    float* dkp = dkv + bi * dkv_bs + tok * d + c0;
    load8(dkp, dk);
    float ds[8], dsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = expf(sc[i] - m[i]) / l[i];
      dk[i] = fmaf(w, gv[i], dk[i]);
      ds[i] = w * gv[i] * (v[i] - pooled[i]);
      dsum += ds[i];
    }
    store8(dkp, dk);
    if (score_width == 1) {
      atomicAdd(dscore + (long long)bi * sq + tok, dsum);
    } else {
      store8(dscore + ((long long)bi * sq + tok) * score_width + c0, ds);
    }
  }
}

cudaError_t launch_compress_bwd(const void* kv, long long kv_bs, const void* score,
                                int score_width, const float* g, long long g_bs, float* dkv,
                                long long dkv_bs, float* dscore, int b, int sq, int d, int ratio,
                                bool bf16, cudaStream_t s) {
  const int n_c = sq / ratio;
  // dscore is written for every token; tokens past the last block and the
  // per-token sums of a shared score start from zero
  cudaError_t e = launch_zero_f32(dscore, (size_t)b * sq * score_width, s);
  if (e != cudaSuccess) return e;
  const long long work = (long long)n_c * (d / 8);
  const int threads = 128;
  dim3 grid((unsigned)((work + threads - 1) / threads), (unsigned)b);
  if (bf16) {
    compress_bwd_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
        (const __nv_bfloat16*)kv, kv_bs, (const __nv_bfloat16*)score, score_width, g, g_bs, dkv,
        dkv_bs, dscore, sq, d, ratio, n_c);
    count_launches(1);
  } else {
    compress_bwd_kernel<float><<<grid, threads, 0, s>>>((const float*)kv, kv_bs,
                                                        (const float*)score, score_width, g, g_bs,
                                                        dkv, dkv_bs, dscore, sq, d, ratio, n_c);
    count_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_compress(const void* kv, long long kv_bs, const void* score, int score_width,
                            void* out, long long out_bs, int b, int sq, int d, int ratio,
                            bool bf16, cudaStream_t s) {
  const int n_c = sq / ratio;
  const long long work = (long long)n_c * (d / 8);
  const int threads = 128;
  dim3 grid((unsigned)((work + threads - 1) / threads), (unsigned)b);
  if (bf16) {
    compress_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
        (const __nv_bfloat16*)kv, kv_bs, (const __nv_bfloat16*)score, score_width,
        (__nv_bfloat16*)out, out_bs, sq, d, ratio, n_c);
    count_launches(1);
  } else {
    compress_kernel<float><<<grid, threads, 0, s>>>((const float*)kv, kv_bs, (const float*)score,
                                                    score_width, (float*)out, out_bs, sq, d,
                                                    ratio, n_c);
    count_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace csa
