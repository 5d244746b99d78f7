// csa_compress_norm_rope / csa_compress_norm_rope_bwd: the compressor with the
// normalization and the rotary embedding of its pooled rows, and the gradient
// of the three.
//
// "Add unfused SBHD compressed sparse attention", compressor review: the
// pooled row is cast once to the storage dtype and then normalized
// (kv = self.norm(kv)); its config fields give the rotary base of compressed
// KV positions (40000).  The library's readings: RMS normalization over the
// d channels with a per-channel weight, in fp32 on the cast pooled row; the
// rotary embedding turns the interleaved pairs (2i, 2i+1) of the last
// rope_dim channels by pos * base^(-2i/rope_dim), with entry j at the
// position of the last token it pools, (j+1)*ratio - 1; the result is cast
// once more.
//
// One warp per pooled row: lane l owns the 8-channel groups l and l + 32
// (d <= 512), so the row's sum of squares and the backward's row dot
// product are warp reductions.  The rotation angles are formed in double
// precision (positions reach 10^5 and more; an fp32 product would lose the
// angle's low bits) and their sine and cosine rounded to fp32 once.
#include "compress_pool.cuh"
#include "csa_common.cuh"
#include "csa_kernels.h"

namespace csa {
namespace {

constexpr int kRowsPerCta = 4;                  // warps per CTA, one pooled row each
constexpr int kMaxGroups = 2;                   // 8-channel groups per lane (d <= 512)

// cos and sin of the rotation of channel pair i (0-based within the rotary
// part) at position pos.
__device__ __forceinline__ void rope_cs(long long pos, int i, int rope_dim, float base, float* c,
                                        float* s) {
  const double theta = exp(-(2.0 * i / rope_dim) * log((double)base));
  double sd, cd;
  sincos((double)pos * theta, &sd, &cd);
  *c = (float)cd;
  *s = (float)sd;
}

// Rotate (or, with sign = -1, rotate back) the rotary pairs among 8 channels
// starting at channel c0.
__device__ __forceinline__ void rope8(float* v, int c0, int d, int rope_dim, float base,
                                      long long pos, float sign) {
  const int r0 = d - rope_dim;
  if (c0 + 8 <= r0) return;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int c = c0 + e;
    if (c < r0) continue;
    float cs, sn;
    rope_cs(pos, (c - r0) / 2, rope_dim, base, &cs, &sn);
    sn *= sign;
    const float a = v[e], b = v[e + 1];
    v[e] = a * cs - b * sn;
    v[e + 1] = a * sn + b * cs;
  }
}

template <typename T>
__device__ __forceinline__ float round_to(float x) {
  return to_f(from_f<T>(x));
}

template <typename T, int R>
__global__ void __launch_bounds__(32 * kRowsPerCta) compress_norm_rope_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ weight, float eps, int rope_dim, float base, T* __restrict__ out,
    long long out_bs, int b, int sq, int d, int ratio, int n_c) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= (long long)b * n_c) return;          // warp-uniform
  const int bi = (int)(row / n_c), j = (int)(row % n_c);
  const int groups = d / 8;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  float x[kMaxGroups][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxGroups; ++k) {
    const int gidx = lane + 32 * k;
    if (gidx >= groups) continue;
    const int c0 = gidx * 8;
    const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
    constexpr int RR = R > 0 ? R : 1;
    float v[RR][8], s[RR][8];
    if constexpr (R > 0) {
#pragma unroll
      for (int t = 0; t < R; ++t) load_token(kvp, scp, t, d, score_width, c0, v[t], s[t]);
    }
    float m[8], l[8], pooled[8];
    pool_block<T, R>(kvp, scp, ratio, d, score_width, c0, v, s, m, l, pooled);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[k][i] = round_to<T>(pooled[i]);           // the pooled row's one cast
      ss = fmaf(x[k][i], x[k][i], ss);
    }
  }
  ss = warp_sum(ss);
  const float rms = sqrtf(ss / (float)d + eps);
  const long long pos = (long long)(j + 1) * ratio - 1;
#pragma unroll
  for (int k = 0; k < kMaxGroups; ++k) {
    const int gidx = lane + 32 * k;
    if (gidx >= groups) continue;
    const int c0 = gidx * 8;
    float y[8], w[8];
    load8(weight + c0, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = x[k][i] / rms * w[i];
    if (rope_dim > 0) rope8(y, c0, d, rope_dim, base, pos, 1.f);
    store8(out + bi * out_bs + (long long)j * d + c0, y);
  }
}

// Backward.  With x the cast pooled row, xh = x / rms, g the gradient of the
// output row and dy = g rotated back:
//   dweight += dy * xh                    (per channel, over all rows)
//   dx = (dy*w - xh * mean(dy*w*xh)) / rms
// and dx flows through the cast unchanged into the pooling backward:
//   dkv_t += w_t dx,  dscore_t = w_t dx (kv_t - pooled)   (as csa_compress_bwd)
template <typename T, int R>
__global__ void __launch_bounds__(32 * kRowsPerCta) compress_norm_rope_bwd_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ weight, float eps, int rope_dim, float base,
    const float* __restrict__ g, long long g_bs, float* __restrict__ dkv, long long dkv_bs,
    float* __restrict__ dscore, float* __restrict__ dweight, int b, int sq, int d, int ratio,
    int n_c) {
  extern __shared__ float s_dw[];                 // [d] this CTA's weight gradient
  for (int c = threadIdx.x; c < d; c += blockDim.x) s_dw[c] = 0.f;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  const int groups = d / 8;
  if (row < (long long)b * n_c) {                 // warp-uniform
    const int bi = (int)(row / n_c), j = (int)(row % n_c);
    const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
    float x[kMaxGroups][8], pooled[kMaxGroups][8], m[kMaxGroups][8], l[kMaxGroups][8];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxGroups; ++k) {
      const int gidx = lane + 32 * k;
      if (gidx >= groups) continue;
      const int c0 = gidx * 8;
      const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
      constexpr int RR = R > 0 ? R : 1;
      float v[RR][8], s[RR][8];
      if constexpr (R > 0) {
#pragma unroll
        for (int t = 0; t < R; ++t) load_token(kvp, scp, t, d, score_width, c0, v[t], s[t]);
      }
      pool_block<T, R>(kvp, scp, ratio, d, score_width, c0, v, s, m[k], l[k], pooled[k]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[k][i] = round_to<T>(pooled[k][i]);
        ss = fmaf(x[k][i], x[k][i], ss);
      }
    }
    ss = warp_sum(ss);
    const float rms = sqrtf(ss / (float)d + eps);
    const long long pos = (long long)(j + 1) * ratio - 1;
    float dxh[kMaxGroups][8];
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxGroups; ++k) {
      const int gidx = lane + 32 * k;
      if (gidx >= groups) continue;
      const int c0 = gidx * 8;
      float dy[8], w[8];
      load8(g + bi * g_bs + (long long)j * d + c0, dy);
      if (rope_dim > 0) rope8(dy, c0, d, rope_dim, base, pos, -1.f);
      load8(weight + c0, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float xh = x[k][i] / rms;
        atomicAdd(&s_dw[c0 + i], dy[i] * xh);
        dxh[k][i] = dy[i] * w[i];
        dot = fmaf(dxh[k][i], xh, dot);
      }
    }
    dot = warp_sum(dot) / (float)d;
#pragma unroll
    for (int k = 0; k < kMaxGroups; ++k) {
      const int gidx = lane + 32 * k;
      if (gidx >= groups) continue;
      const int c0 = gidx * 8;
      float dx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) dx[i] = (dxh[k][i] - x[k][i] / rms * dot) / rms;
      // the pooling backward of this group's channels
      const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
      float* dkp = dkv + bi * dkv_bs + (long long)j * ratio * d + c0;
      for (int t = 0; t < ratio; ++t) {
        float vt[8], st[8], dt[8];
        load_token(kvp, scp, t, d, score_width, c0, vt, st);
        load8(dkp + (long long)t * d, dt);
        const long long tok = (long long)j * ratio + t;
        float ds[8], dsum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float wt = expf(st[i] - m[k][i]) / l[k][i];
          dt[i] = fmaf(wt, dx[i], dt[i]);
          ds[i] = wt * dx[i] * (vt[i] - pooled[k][i]);
          dsum += ds[i];
        }
        store8(dkp + (long long)t * d, dt);
        if (score_width == 1)
          atomicAdd(dscore + (long long)bi * sq + tok, dsum);
        else
          store8(dscore + ((long long)bi * sq + tok) * score_width + c0, ds);
      }
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += blockDim.x) atomicAdd(&dweight[c], s_dw[c]);
}

// Tail tokens (sq % ratio of them) get a zero score gradient (per-channel
// scores; a shared score is zeroed before the launch).
__global__ void zero_tail_rows(float* __restrict__ dscore, int b, int sq, int d, int t0) {
  const int rows = sq - t0;
  const long long n = (long long)b * rows * d;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / d;
    const int bi = (int)(r / rows), t = t0 + (int)(r % rows);
    dscore[((long long)bi * sq + t) * d + i % d] = 0.f;
  }
}

}  // namespace

cudaError_t launch_compress_norm_rope(const void* kv, long long kv_bs, const void* score,
                                      int score_width, const float* weight, float eps,
                                      int rope_dim, float base, void* out, long long out_bs,
                                      int b, int sq, int d, int ratio, bool bf16,
                                      cudaStream_t s) {
  const int n_c = sq / ratio;
  const long long rows = (long long)b * n_c;
  const unsigned grid = (unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta);
#define CSA_NR(TT, RR)                                                                         \
  compress_norm_rope_kernel<TT, RR><<<grid, 32 * kRowsPerCta, 0, s>>>(                         \
      (const TT*)kv, kv_bs, (const TT*)score, score_width, weight, eps, rope_dim, base,        \
      (TT*)out, out_bs, b, sq, d, ratio, n_c)
  if (bf16) {
    if (ratio == 4) CSA_NR(__nv_bfloat16, 4); else CSA_NR(__nv_bfloat16, 0);
  } else {
    if (ratio == 4) CSA_NR(float, 4); else CSA_NR(float, 0);
  }
#undef CSA_NR
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_compress_norm_rope_bwd(const void* kv, long long kv_bs, const void* score,
                                          int score_width, const float* weight, float eps,
                                          int rope_dim, float base, const float* g,
                                          long long g_bs, float* dkv, long long dkv_bs,
                                          float* dscore, float* dweight, int b, int sq, int d,
                                          int ratio, bool bf16, cudaStream_t s) {
  const int n_c = sq / ratio;
  cudaError_t e = launch_zero_f32(dweight, (size_t)d, s);
  if (e != cudaSuccess) return e;
  if (score_width == 1) {
    e = launch_zero_f32(dscore, (size_t)b * sq, s);
    if (e != cudaSuccess) return e;
  } else if (n_c * ratio < sq) {
    zero_tail_rows<<<64, 256, 0, s>>>(dscore, b, sq, d, n_c * ratio);
    count_launches(1);
  }
  const long long rows = (long long)b * n_c;
  const unsigned grid = (unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta);
  const size_t smem = (size_t)d * sizeof(float);
#define CSA_NRB(TT, RR)                                                                        \
  compress_norm_rope_bwd_kernel<TT, RR><<<grid, 32 * kRowsPerCta, smem, s>>>(                  \
      (const TT*)kv, kv_bs, (const TT*)score, score_width, weight, eps, rope_dim, base, g,     \
      g_bs, dkv, dkv_bs, dscore, dweight, b, sq, d, ratio, n_c)
  if (bf16) {
    if (ratio == 4) CSA_NRB(__nv_bfloat16, 4); else CSA_NRB(__nv_bfloat16, 0);
  } else {
    if (ratio == 4) CSA_NRB(float, 4); else CSA_NRB(float, 0);
  }
#undef CSA_NRB
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
