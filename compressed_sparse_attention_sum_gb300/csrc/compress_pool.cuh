// Pooling helpers shared by the compressor kernels (compress.cu,
// compress_norm_rope.cu): the softmax-weighted pooling of one block's tokens
// for 8 consecutive channels, in fp32 ("Add unfused SBHD compressed sparse
// attention", compressor review).
#pragma once

#include "csa_common.cuh"

namespace csa {

// 8 channels of token t of a block: kv row and the pooling score (the score is
// broadcast over the channels when one score drives the whole row)
template <typename T>
__device__ __forceinline__ void load_token(const T* kvp, const T* scp, int t, int d,
                                           int score_width, int c0, float* v, float* s) {
  load8(kvp + (long long)t * d, v);
  if (score_width == 1) {
    const float s1 = to_f(scp[t]);
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = s1;
  } else {
    load8(scp + (long long)t * score_width + c0, s);
  }
}

// Per-channel softmax statistics of a block (running max m, sum l) and the
// pooled value sum_t w_t kv_t.  R > 0: compile-time ratio, the block is held
// in registers (v, s filled by the caller); R == 0: runtime ratio, online.
template <typename T, int R>
__device__ __forceinline__ void pool_block(const T* kvp, const T* scp, int ratio, int d,
                                           int score_width, int c0, float (*v)[8],
                                           float (*s)[8], float* m, float* l, float* pooled) {
  if constexpr (R > 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float mx = s[0][i];
#pragma unroll
      for (int t = 1; t < R; ++t) mx = fmaxf(mx, s[t][i]);
      float sum = 0.f, acc = 0.f;
#pragma unroll
      for (int t = 0; t < R; ++t) {
        const float e = expf(s[t][i] - mx);
        sum += e;
        acc = fmaf(e, v[t][i], acc);
      }
      m[i] = mx;
      l[i] = sum;
      pooled[i] = acc / sum;
    }
  } else {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { m[i] = -INFINITY; l[i] = 0.f; acc[i] = 0.f; }
    for (int t = 0; t < ratio; ++t) {
      float vt[8], st[8];
      load_token(kvp, scp, t, d, score_width, c0, vt, st);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float mn = fmaxf(m[i], st[i]);
        const float alpha = expf(m[i] - mn);  // 0 on the first token (m = -inf)
        const float e = expf(st[i] - mn);
        l[i] = l[i] * alpha + e;
        acc[i] = acc[i] * alpha + e * vt[i];
        m[i] = mn;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) pooled[i] = acc[i] / l[i];
  }
}

}  // namespace csa
