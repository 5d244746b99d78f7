// csa_compress / csa_compress_bwd: softmax-weighted pooling of `ratio`
// consecutive KV tokens, and its gradient.
//
// "Add unfused SBHD compressed sparse attention" (Megatron-LM PR #6400),
// compressor review: the softmax over the block's tokens, the products and
// the sum stay in fp32 and the pooled row is cast once to the storage dtype.
//
// HBM-bound: each kv and score element is read once and each pooled element
// written once.  One thread owns 8 consecutive channels of one block.  For
// ratio 4 (the CSA ratio) the thread loads the whole block before any
// arithmetic, so one memory latency covers it; other small ratios walk the
// tokens with an online (running max) softmax, reading the scores in one
// pass; ratios of 16 and more (HCA: 128) split each block's tokens over the
// threads of a CTA and merge the partial softmax statistics.
#include "compress_pool.cuh"
#include "csa_common.cuh"
#include "csa_kernels.h"

namespace csa {

template <typename T, int R>
__global__ void __launch_bounds__(64) compress_kernel(const T* __restrict__ kv, long long kv_bs,
                                                      const T* __restrict__ score,
                                                      int score_width, T* __restrict__ out,
                                                      long long out_bs, int sq, int d, int ratio,
                                                      int n_c) {
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int bi = blockIdx.y;
  if (gid >= (long long)n_c * groups) return;
  const int j = (int)(gid / groups);
  const int c0 = (int)(gid % groups) * 8;
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  constexpr int RR = R > 0 ? R : 1;
  float v[RR][8], s[RR][8];
  if constexpr (R > 0) {
#pragma unroll
    for (int t = 0; t < R; ++t) load_token(kvp, scp, t, d, score_width, c0, v[t], s[t]);
  }
  float m[8], l[8], r[8];
  pool_block<T, R>(kvp, scp, ratio, d, score_width, c0, v, s, m, l, r);
  store8(out + bi * out_bs + (long long)j * d + c0, r);
}

// Backward of the pooling.  With w_t the softmax weights of a block and
// channel, pooled = sum_t w_t kv_t and g = dL/dpooled:
//   dkv_t    += w_t g                      (accumulated: the raw rows also get
//                                           the attention's gradient)
//   dscore_t  = w_t g (kv_t - pooled)      (per channel; summed over channels
//                                           when one score drives all channels)
// Tokens past the last complete block get no kv gradient and zero dscore; with
// a per-channel score the threads past the last block write those zeros.
template <typename T, int R>
__global__ void __launch_bounds__(64) compress_bwd_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ g, long long g_bs, float* __restrict__ dkv, long long dkv_bs,
    float* __restrict__ dscore, int sq, int d, int ratio, int n_c) {
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int bi = blockIdx.y;
  if (gid >= (long long)n_c * groups) {
    if (score_width == 1) return;  // zeroed before the launch
    const long long tok = (long long)n_c * ratio + (gid - (long long)n_c * groups) / groups;
    if (tok >= sq) return;
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    store8(dscore + ((long long)bi * sq + tok) * score_width + (gid % groups) * 8, z);
    return;
  }
  const int j = (int)(gid / groups);
  const int c0 = (int)(gid % groups) * 8;
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  float* dkp = dkv + bi * dkv_bs + (long long)j * ratio * d + c0;
  float gv[8];
  load8(g + bi * g_bs + (long long)j * d + c0, gv);
  constexpr int RR = R > 0 ? R : 1;
  float v[RR][8], s[RR][8], dk[RR][8];
  if constexpr (R > 0) {
    // everything the block needs, before any arithmetic
#pragma unroll
    for (int t = 0; t < R; ++t) {
      load_token(kvp, scp, t, d, score_width, c0, v[t], s[t]);
      load8(dkp + (long long)t * d, dk[t]);
    }
  }
  float m[8], l[8], pooled[8];
  pool_block<T, R>(kvp, scp, ratio, d, score_width, c0, v, s, m, l, pooled);
  const int nt = R > 0 ? R : ratio;
#pragma unroll(R > 0 ? R : 1)
  for (int t = 0; t < nt; ++t) {
    float vt[8], st[8], dt[8];
    if constexpr (R > 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) { vt[i] = v[t][i]; st[i] = s[t][i]; dt[i] = dk[t][i]; }
    } else {
      load_token(kvp, scp, t, d, score_width, c0, vt, st);
      load8(dkp + (long long)t * d, dt);
    }
    const long long tok = (long long)j * ratio + t;
    float ds[8], dsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = expf(st[i] - m[i]) / l[i];
      dt[i] = fmaf(w, gv[i], dt[i]);
      ds[i] = w * gv[i] * (vt[i] - pooled[i]);
      dsum += ds[i];
    }
    store8(dkp + (long long)t * d, dt);
    if (score_width == 1) {
      atomicAdd(dscore + (long long)bi * sq + tok, dsum);
    } else {
      store8(dscore + ((long long)bi * sq + tok) * score_width + c0, ds);
    }
  }
}

// Overlapping compression: entry j pools the coff blocks ending with block j,
// tokens [max(0, (j + 1 - coff) r), (j + 1) r), with one softmax over the
// window ("Add unfused SBHD compressed sparse attention", compressor review:
// coff = 1 is the non-overlapping case).  Online softmax over the window.
template <typename T>
__global__ void __launch_bounds__(64) compress_overlap_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    T* __restrict__ out, long long out_bs, int sq, int d, int ratio, int n_c, int coff) {
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int bi = blockIdx.y;
  if (gid >= (long long)n_c * groups) return;
  const int j = (int)(gid / groups);
  const int c0 = (int)(gid % groups) * 8;
  const int t0 = max(0, (j + 1 - coff) * ratio);
  const T* kvp = kv + bi * kv_bs + (long long)t0 * d + c0;
  const T* scp = score + ((long long)bi * sq + t0) * score_width;
  float v[1][8], s[1][8], m[8], l[8], r[8];
  pool_block<T, 0>(kvp, scp, (j + 1) * ratio - t0, d, score_width, c0, v, s, m, l, r);
  store8(out + bi * out_bs + (long long)j * d + c0, r);
}

// Its backward.  The thread of block j owns the block's ratio tokens, which
// lie in the windows of entries j .. j + C - 1; it forms those windows'
// softmax statistics and pooled rows first, then sums the windows'
// contributions per token, so every token is written by one thread.
template <typename T, int C>
__global__ void __launch_bounds__(64) compress_overlap_bwd_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ g, long long g_bs, float* __restrict__ dkv, long long dkv_bs,
    float* __restrict__ dscore, int sq, int d, int ratio, int n_c) {
  const int groups = d / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int bi = blockIdx.y;
  if (gid >= (long long)n_c * groups) {
    if (score_width == 1) return;  // zeroed before the launch
    const long long tok = (long long)n_c * ratio + (gid - (long long)n_c * groups) / groups;
    if (tok >= sq) return;
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    store8(dscore + ((long long)bi * sq + tok) * score_width + (gid % groups) * 8, z);
    return;
  }
  const int j = (int)(gid / groups);
  const int c0 = (int)(gid % groups) * 8;
  const T* kvb = kv + bi * kv_bs + c0;
  const T* scb = score + (long long)bi * sq * score_width;
  float m[C][8], l[C][8], pooled[C][8], gv[C][8];
#pragma unroll
  for (int k = 0; k < C; ++k) {
    const int w = j + k;
    if (w >= n_c) continue;
    const int t0 = max(0, (w + 1 - C) * ratio);
    float v[1][8], s[1][8];
    pool_block<T, 0>(kvb + (long long)t0 * d, scb + (long long)t0 * score_width,
                     (w + 1) * ratio - t0, d, score_width, c0, v, s, m[k], l[k], pooled[k]);
    load8(g + bi * g_bs + (long long)w * d + c0, gv[k]);
  }
  float* dkp = dkv + bi * dkv_bs + (long long)j * ratio * d + c0;
  for (int t = 0; t < ratio; ++t) {
    const long long tok = (long long)j * ratio + t;
    float vt[8], st[8], dt[8], ds[8];
    load_token(kvb + (long long)j * ratio * d, scb + (long long)j * ratio * score_width, t, d,
               score_width, c0, vt, st);
    load8(dkp + (long long)t * d, dt);
#pragma unroll
    for (int i = 0; i < 8; ++i) ds[i] = 0.f;
#pragma unroll
    for (int k = 0; k < C; ++k) {
      if (j + k >= n_c) continue;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float w = expf(st[i] - m[k][i]) / l[k][i];
        dt[i] = fmaf(w, gv[k][i], dt[i]);
        ds[i] = fmaf(w * gv[k][i], vt[i] - pooled[k][i], ds[i]);
      }
    }
    store8(dkp + (long long)t * d, dt);
    if (score_width == 1) {
      float dsum = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) dsum += ds[i];
      atomicAdd(dscore + (long long)bi * sq + tok, dsum);
    } else {
      store8(dscore + ((long long)bi * sq + tok) * score_width + c0, ds);
    }
  }
}

// Large ratios (the HCA ratio 128): one CTA per block, whose threads split
// the block's tokens into TS ranges as well as its channels (8 per thread).
// Each thread forms the online softmax of its tokens; the partial (max, sum,
// weighted sum) triples are merged in shared memory.  A thread per (block,
// 8 channels) walking all `ratio` tokens, as above, would leave a few
// thousand threads each waiting on `ratio` dependent loads in turn.
constexpr int kSplitThreads = 256;
constexpr int kSplitMinRatio = 16;

template <typename T>
__device__ __forceinline__ void split_partial(const T* kvp, const T* scp, int d, int score_width,
                                              int c0, int t_lo, int t_hi, float* m, float* l,
                                              float* acc) {
#pragma unroll
  for (int i = 0; i < 8; ++i) { m[i] = -INFINITY; l[i] = 0.f; acc[i] = 0.f; }
  for (int t = t_lo; t < t_hi; ++t) {
    float vt[8], st[8];
    load_token(kvp, scp, t, d, score_width, c0, vt, st);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float mn = fmaxf(m[i], st[i]);
      const float alpha = expf(m[i] - mn);    // 0 on the first token (m = -inf)
      const float e = expf(st[i] - mn);
      l[i] = l[i] * alpha + e;
      acc[i] = acc[i] * alpha + e * vt[i];
      m[i] = mn;
    }
  }
}

// The block's statistics per channel: the TS partials of this CTA merged by
// the threads of token range 0 into (M, L, pooled), left in shared memory
// (sm[0..3*groups*8)) for every thread.  kvp points at channel 0 of the
// block's first token.
template <typename T>
__device__ __forceinline__ void split_stats(const T* kvp, const T* scp, int d, int score_width,
                                            int ratio, float* sm, int groups, int TS, int cg,
                                            int ts) {
  const int per = (ratio + TS - 1) / TS;
  float m[8], l[8], acc[8];
  const int t_lo = min(ratio, ts * per), t_hi = min(ratio, t_lo + per);
  if (ts < TS) {
    split_partial(kvp + cg * 8, scp, d, score_width, cg * 8, t_lo, t_hi, m, l, acc);
    float* pm = sm + ((size_t)ts * groups + cg) * 24;
#pragma unroll
    for (int i = 0; i < 8; ++i) { pm[i] = m[i]; pm[8 + i] = l[i]; pm[16 + i] = acc[i]; }
  }
  __syncthreads();
  float M[8], L[8], A[8];
  if (ts == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) { M[i] = -INFINITY; L[i] = 0.f; A[i] = 0.f; }
    for (int k = 0; k < TS; ++k) {
      const float* pm = sm + ((size_t)k * groups + cg) * 24;
#pragma unroll
      for (int i = 0; i < 8; ++i) M[i] = fmaxf(M[i], pm[i]);
    }
    for (int k = 0; k < TS; ++k) {
      const float* pm = sm + ((size_t)k * groups + cg) * 24;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float f = expf(pm[i] - M[i]);   // 0 for an empty range (m = -inf)
        L[i] = fmaf(pm[8 + i], f, L[i]);
        A[i] = fmaf(pm[16 + i], f, A[i]);
      }
    }
  }
  __syncthreads();              // every partial has been read
  if (ts == 0) {
    float* st = sm + (size_t)cg * 24;
#pragma unroll
    for (int i = 0; i < 8; ++i) { st[i] = M[i]; st[8 + i] = L[i]; st[16 + i] = A[i] / L[i]; }
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kSplitThreads) compress_split_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    T* __restrict__ out, long long out_bs, int sq, int d, int ratio) {
  extern __shared__ float sm_split[];
  const int groups = d / 8, TS = kSplitThreads / groups;
  const int j = blockIdx.x, bi = blockIdx.y;
  const int cg = threadIdx.x % groups, ts = threadIdx.x / groups;
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  split_stats(kvp, scp, d, score_width, ratio, sm_split, groups, TS, cg, ts);
  if (ts == 0) store8(out + bi * out_bs + (long long)j * d + cg * 8, sm_split + cg * 24 + 16);
}

// Its backward: the block's statistics as above, then every thread adds
// w_t g to its tokens' dkv rows and writes their score gradients (the CTA
// past the last block writes the zero score gradient of the tail tokens).
template <typename T>
__global__ void __launch_bounds__(kSplitThreads) compress_bwd_split_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ g, long long g_bs, float* __restrict__ dkv, long long dkv_bs,
    float* __restrict__ dscore, int sq, int d, int ratio, int n_c) {
  extern __shared__ float sm_split[];
  const int groups = d / 8, TS = kSplitThreads / groups;
  const int j = blockIdx.x, bi = blockIdx.y;
  const int cg = threadIdx.x % groups, ts = threadIdx.x / groups;
  if (j >= n_c) {             // tail tokens: zero score gradient (per-channel scores)
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int t = n_c * ratio + ts; ts < TS && t < sq; t += TS)
      store8(dscore + ((long long)bi * sq + t) * score_width + cg * 8, z);
    return;
  }
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  split_stats(kvp, scp, d, score_width, ratio, sm_split, groups, TS, cg, ts);
  if (ts >= TS) return;
  const int c0 = cg * 8;
  float M[8], L[8], P[8], gv[8];
  const float* st = sm_split + cg * 24;
#pragma unroll
  for (int i = 0; i < 8; ++i) { M[i] = st[i]; L[i] = st[8 + i]; P[i] = st[16 + i]; }
  load8(g + bi * g_bs + (long long)j * d + c0, gv);
  const int per = (ratio + TS - 1) / TS;
  const int t_lo = min(ratio, ts * per), t_hi = min(ratio, t_lo + per);
  float* dkp = dkv + bi * dkv_bs + (long long)j * ratio * d + c0;
  for (int t = t_lo; t < t_hi; ++t) {
    float vt[8], sv[8], dt[8];
    load_token(kvp + c0, scp, t, d, score_width, c0, vt, sv);
    load8(dkp + (long long)t * d, dt);
    float ds[8], dsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = expf(sv[i] - M[i]) / L[i];
      dt[i] = fmaf(w, gv[i], dt[i]);
      ds[i] = w * gv[i] * (vt[i] - P[i]);
      dsum += ds[i];
    }
    store8(dkp + (long long)t * d, dt);
    const long long tok = (long long)j * ratio + t;
    if (score_width == 1)
      atomicAdd(dscore + (long long)bi * sq + tok, dsum);
    else
      store8(dscore + ((long long)bi * sq + tok) * score_width + c0, ds);
  }
}

namespace {
constexpr int kCompressThreads = 64;

size_t split_smem(int d) {
  const int groups = d / 8;
  return (size_t)(kSplitThreads / groups) * groups * 24 * sizeof(float);
}

template <typename T, int R>
void compress_fwd_t(const void* kv, long long kv_bs, const void* score, int score_width,
                    void* out, long long out_bs, int b, int sq, int d, int ratio, cudaStream_t s) {
  const int n_c = sq / ratio;
  if (R == 0 && ratio >= kSplitMinRatio) {
    compress_split_kernel<T><<<dim3((unsigned)n_c, (unsigned)b), kSplitThreads, split_smem(d),
                               s>>>((const T*)kv, kv_bs, (const T*)score, score_width, (T*)out,
                                    out_bs, sq, d, ratio);
    count_launches(1);
    return;
  }
  const long long work = (long long)n_c * (d / 8);
  dim3 grid((unsigned)((work + kCompressThreads - 1) / kCompressThreads), (unsigned)b);
  compress_kernel<T, R><<<grid, kCompressThreads, 0, s>>>((const T*)kv, kv_bs, (const T*)score,
                                                          score_width, (T*)out, out_bs, sq, d,
                                                          ratio, n_c);
  count_launches(1);
}

template <typename T, int R>
void compress_bwd_t(const void* kv, long long kv_bs, const void* score, int score_width,
                    const float* g, long long g_bs, float* dkv, long long dkv_bs, float* dscore,
                    int b, int sq, int d, int ratio, cudaStream_t s) {
  const int n_c = sq / ratio;
  const int tail = score_width == 1 ? 0 : sq - n_c * ratio;
  if (R == 0 && ratio >= kSplitMinRatio) {
    const unsigned nx = (unsigned)(n_c + (tail > 0 ? 1 : 0));
    compress_bwd_split_kernel<T><<<dim3(nx, (unsigned)b), kSplitThreads, split_smem(d), s>>>(
        (const T*)kv, kv_bs, (const T*)score, score_width, g, g_bs, dkv, dkv_bs, dscore, sq, d,
        ratio, n_c);
    count_launches(1);
    return;
  }
  const long long work = (long long)(n_c + tail) * (d / 8);
  if (work == 0) return;
  dim3 grid((unsigned)((work + kCompressThreads - 1) / kCompressThreads), (unsigned)b);
  compress_bwd_kernel<T, R><<<grid, kCompressThreads, 0, s>>>(
      (const T*)kv, kv_bs, (const T*)score, score_width, g, g_bs, dkv, dkv_bs, dscore, sq, d,
      ratio, n_c);
  count_launches(1);
}
}  // namespace

cudaError_t launch_compress_bwd(const void* kv, long long kv_bs, const void* score,
                                int score_width, const float* g, long long g_bs, float* dkv,
                                long long dkv_bs, float* dscore, int b, int sq, int d, int ratio,
                                bool bf16, cudaStream_t s) {
  if (score_width == 1) {
    // the per-token sums of a shared score (and the tail) start from zero
    cudaError_t e = launch_zero_f32(dscore, (size_t)b * sq, s);
    if (e != cudaSuccess) return e;
  }
  if (bf16) {
    if (ratio == 4)
      compress_bwd_t<__nv_bfloat16, 4>(kv, kv_bs, score, score_width, g, g_bs, dkv, dkv_bs,
                                       dscore, b, sq, d, ratio, s);
    else
      compress_bwd_t<__nv_bfloat16, 0>(kv, kv_bs, score, score_width, g, g_bs, dkv, dkv_bs,
                                       dscore, b, sq, d, ratio, s);
  } else {
    if (ratio == 4)
      compress_bwd_t<float, 4>(kv, kv_bs, score, score_width, g, g_bs, dkv, dkv_bs, dscore, b,
                               sq, d, ratio, s);
    else
      compress_bwd_t<float, 0>(kv, kv_bs, score, score_width, g, g_bs, dkv, dkv_bs, dscore, b,
                               sq, d, ratio, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_compress(const void* kv, long long kv_bs, const void* score, int score_width,
                            void* out, long long out_bs, int b, int sq, int d, int ratio,
                            bool bf16, cudaStream_t s) {
  if (bf16) {
    if (ratio == 4)
      compress_fwd_t<__nv_bfloat16, 4>(kv, kv_bs, score, score_width, out, out_bs, b, sq, d,
                                       ratio, s);
    else
      compress_fwd_t<__nv_bfloat16, 0>(kv, kv_bs, score, score_width, out, out_bs, b, sq, d,
                                       ratio, s);
  } else {
    if (ratio == 4)
      compress_fwd_t<float, 4>(kv, kv_bs, score, score_width, out, out_bs, b, sq, d, ratio, s);
    else
      compress_fwd_t<float, 0>(kv, kv_bs, score, score_width, out, out_bs, b, sq, d, ratio, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_compress_overlap(const void* kv, long long kv_bs, const void* score,
                                    int score_width, void* out, long long out_bs, int b, int sq,
                                    int d, int ratio, int coff, bool bf16, cudaStream_t s) {
  if (coff == 1)
    return launch_compress(kv, kv_bs, score, score_width, out, out_bs, b, sq, d, ratio, bf16, s);
  const int n_c = sq / ratio;
  const long long work = (long long)n_c * (d / 8);
  dim3 grid((unsigned)((work + kCompressThreads - 1) / kCompressThreads), (unsigned)b);
  if (bf16)
    compress_overlap_kernel<__nv_bfloat16><<<grid, kCompressThreads, 0, s>>>(
        (const __nv_bfloat16*)kv, kv_bs, (const __nv_bfloat16*)score, score_width,
        (__nv_bfloat16*)out, out_bs, sq, d, ratio, n_c, coff);
  else
    compress_overlap_kernel<float><<<grid, kCompressThreads, 0, s>>>(
        (const float*)kv, kv_bs, (const float*)score, score_width, (float*)out, out_bs, sq, d,
        ratio, n_c, coff);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_compress_overlap_bwd(const void* kv, long long kv_bs, const void* score,
                                        int score_width, const float* g, long long g_bs,
                                        float* dkv, long long dkv_bs, float* dscore, int b,
                                        int sq, int d, int ratio, int coff, bool bf16,
                                        cudaStream_t s) {
  if (coff == 1)
    return launch_compress_bwd(kv, kv_bs, score, score_width, g, g_bs, dkv, dkv_bs, dscore, b,
                               sq, d, ratio, bf16, s);
  if (coff != 2) return cudaErrorInvalidValue;
  if (score_width == 1) {
    cudaError_t e = launch_zero_f32(dscore, (size_t)b * sq, s);
    if (e != cudaSuccess) return e;
  }
  const int n_c = sq / ratio;
  const int tail = score_width == 1 ? 0 : sq - n_c * ratio;
  const long long work = (long long)(n_c + tail) * (d / 8);
  if (work == 0) return cudaSuccess;
  dim3 grid((unsigned)((work + kCompressThreads - 1) / kCompressThreads), (unsigned)b);
  if (bf16)
    compress_overlap_bwd_kernel<__nv_bfloat16, 2><<<grid, kCompressThreads, 0, s>>>(
        (const __nv_bfloat16*)kv, kv_bs, (const __nv_bfloat16*)score, score_width, g, g_bs, dkv,
        dkv_bs, dscore, sq, d, ratio, n_c);
  else
    compress_overlap_bwd_kernel<float, 2><<<grid, kCompressThreads, 0, s>>>(
        (const float*)kv, kv_bs, (const float*)score, score_width, g, g_bs, dkv, dkv_bs, dscore,
        sq, d, ratio, n_c);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
