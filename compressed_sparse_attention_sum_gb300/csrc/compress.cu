// csa_compress: softmax-weighted pooling of `ratio` consecutive KV tokens.
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
