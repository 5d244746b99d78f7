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
// threads of a CTA and reduce the block's softmax statistics across them.
#include "compress_pool.cuh"
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"

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

// Large ratios (the HCA ratio 128): a CTA per (block, batch, channel slice).
// A slice is G groups of 8 channels (G the largest power of two dividing d/8,
// at most 8: C = 8G channels); the CTA's 256 threads form TS = 256/G token
// lanes of G threads, token lane ts taking the block's tokens ts, ts + TS, ...
// Every thread loads its first kSplitCache tokens before any arithmetic, so
// one memory latency covers the block.  The softmax statistics then come from
// two reductions, each over a warp's lanes by shuffles and over the CTA's
// warps in shared memory: the block maximum M per channel, then the sums of
// e_t = 2^(s_t log2(e) - M log2(e)) and of e_t kv_t under that common maximum
// (one exponential per element, no rescaling of partial sums).
constexpr int kSplitThreads = 256;
constexpr int kSplitWarps = kSplitThreads / 32;
constexpr int kSplitCache = 4;
constexpr int kSplitMinRatio = 16;

int split_slice_groups(int groups) {
  int g = 1;
  while (g < 8 && groups % (2 * g) == 0) g *= 2;
  return g;
}

struct SplitShared {
  float red[kSplitWarps][2][64];   // per-warp partial maxima / sums of the C channels
  float M2[64], L[64], P[64];      // M log2(e), sum of e_t, pooled value
};

template <typename T>
__device__ __forceinline__ void load_score8(const T* scp, int t, int score_width, int c0, float* s) {
  if (score_width == 1) {
    const float s1 = to_f(scp[t]);
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = s1;
  } else {
    load8(scp + (long long)t * score_width + c0, s);
  }
}

// The block's statistics for the thread's 8 channels (c0..c0+7) and, in S, for
// the CTA's C channels.  kvp points at channel c0 of the block's first token,
// scp at the block's first score.  On return vc/sc hold the kv and score values
// of the thread's first min(n_my, kSplitCache) tokens.
template <typename T>
__device__ __forceinline__ void split_block_stats(const T* kvp, const T* scp, int d,
                                                  int score_width, int TS, int G, int ts,
                                                  int cgl, int c0, int n_my,
                                                  float (&vc)[kSplitCache][8],
                                                  float (&sc)[kSplitCache][8], SplitShared& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, C = 8 * G;
#pragma unroll
  for (int k = 0; k < kSplitCache; ++k)
    if (k < n_my) load_token(kvp, scp, ts + k * TS, d, score_width, c0, vc[k], sc[k]);
  float r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = -INFINITY;
#pragma unroll
  for (int k = 0; k < kSplitCache; ++k)
    if (k < n_my) {
#pragma unroll
      for (int i = 0; i < 8; ++i) r[i] = fmaxf(r[i], sc[k][i]);
    }
  for (int k = kSplitCache; k < n_my; ++k) {
    float st[8];
    load_score8(scp, ts + k * TS, score_width, c0, st);
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = fmaxf(r[i], st[i]);
  }
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = fmaxf(r[i], __shfl_xor_sync(0xffffffffu, r[i], o));
  }
  if (lane < G) {
#pragma unroll
    for (int i = 0; i < 8; ++i) S.red[warp][0][cgl * 8 + i] = r[i];
  }
  __syncthreads();
  if (tid < C) {
    float m = S.red[0][0][tid];
#pragma unroll
    for (int w = 1; w < kSplitWarps; ++w) m = fmaxf(m, S.red[w][0][tid]);
    S.M2[tid] = m * kLog2e;
  }
  __syncthreads();
  float m2[8], l[8], a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) { m2[i] = S.M2[cgl * 8 + i]; l[i] = 0.f; a[i] = 0.f; }
#pragma unroll
  for (int k = 0; k < kSplitCache; ++k)
    if (k < n_my) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float e = umma::ex2(fmaf(sc[k][i], kLog2e, -m2[i]));
        l[i] += e;
        a[i] = fmaf(e, vc[k][i], a[i]);
      }
    }
  for (int k = kSplitCache; k < n_my; ++k) {
    float vt[8], st[8];
    load_token(kvp, scp, ts + k * TS, d, score_width, c0, vt, st);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float e = umma::ex2(fmaf(st[i], kLog2e, -m2[i]));
      l[i] += e;
      a[i] = fmaf(e, vt[i], a[i]);
    }
  }
  for (int o = G; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], o);
      a[i] += __shfl_xor_sync(0xffffffffu, a[i], o);
    }
  }
  if (lane < G) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      S.red[warp][0][cgl * 8 + i] = l[i];
      S.red[warp][1][cgl * 8 + i] = a[i];
    }
  }
  __syncthreads();
  if (tid < C) {
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kSplitWarps; ++w) { L += S.red[w][0][tid]; A += S.red[w][1][tid]; }
    S.L[tid] = L;
    S.P[tid] = A / L;
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kSplitThreads) compress_split_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    T* __restrict__ out, long long out_bs, int sq, int d, int ratio, int G) {
  __shared__ SplitShared S;
  const int TS = kSplitThreads / G, cgl = threadIdx.x % G, ts = threadIdx.x / G;
  const int j = blockIdx.x, bi = blockIdx.y, cb = blockIdx.z * G * 8, c0 = cb + cgl * 8;
  const int n_my = ts < ratio ? (ratio - 1 - ts) / TS + 1 : 0;
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  float vc[kSplitCache][8], sc[kSplitCache][8];
  split_block_stats(kvp, scp, d, score_width, TS, G, ts, cgl, c0, n_my, vc, sc, S);
  if (threadIdx.x < 8 * G)
    out[bi * out_bs + (long long)j * d + cb + threadIdx.x] = from_f<T>(S.P[threadIdx.x]);
}

// Its backward: the block's statistics as above, then every thread adds
// w_t g to its tokens' dkv rows (fetched into shared memory at the start, so
// their latency overlaps the statistics) and writes their score gradients;
// with one score per token the G lanes of a token sum theirs before one atomic
// add.  The CTAs past the last block write the zero score gradient of the tail
// tokens (per-channel scores).
template <typename T>
__global__ void __launch_bounds__(kSplitThreads, 2) compress_bwd_split_kernel(
    const T* __restrict__ kv, long long kv_bs, const T* __restrict__ score, int score_width,
    const float* __restrict__ g, long long g_bs, float* __restrict__ dkv, long long dkv_bs,
    float* __restrict__ dscore, int sq, int d, int ratio, int n_c, int G) {
  __shared__ SplitShared S;
  __shared__ __align__(16) float dk_s[kSplitCache][2][kSplitThreads][4];
  const int tid = threadIdx.x, lane = tid & 31;
  const int TS = kSplitThreads / G, cgl = tid % G, ts = tid / G;
  const int j = blockIdx.x, bi = blockIdx.y, cb = blockIdx.z * G * 8, c0 = cb + cgl * 8;
  if (j >= n_c) {
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int t = n_c * ratio + ts; t < sq; t += TS)
      store8(dscore + ((long long)bi * sq + t) * score_width + c0, z);
    return;
  }
  const int n_my = ts < ratio ? (ratio - 1 - ts) / TS + 1 : 0;
  float* dkp = dkv + bi * dkv_bs + (long long)j * ratio * d + c0;
#pragma unroll
  for (int k = 0; k < kSplitCache; ++k)
    if (k < n_my) {
      const float* src = dkp + (long long)(ts + k * TS) * d;
      umma::cp_async_16(&dk_s[k][0][tid][0], src);
      umma::cp_async_16(&dk_s[k][1][tid][0], src + 4);
    }
  float gv[8];
  load8(g + bi * g_bs + (long long)j * d + c0, gv);
  const T* kvp = kv + bi * kv_bs + (long long)j * ratio * d + c0;
  const T* scp = score + ((long long)bi * sq + (long long)j * ratio) * score_width;
  float vc[kSplitCache][8], sc[kSplitCache][8];
  split_block_stats(kvp, scp, d, score_width, TS, G, ts, cgl, c0, n_my, vc, sc, S);
  // w_t = 2^(s_t log2(e) - b2) with b2 = M log2(e) + log2(L)
  float b2[8], P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    b2[i] = S.M2[cgl * 8 + i] + log2f(S.L[cgl * 8 + i]);
    P[i] = S.P[cgl * 8 + i];
  }
  umma::cp_async_wait_all_();
  const unsigned gmask = ((1u << G) - 1u) << (lane & ~(G - 1));
  float* dsp = dscore + ((long long)bi * sq + (long long)j * ratio) * score_width;
  auto grad = [&](int t, const float* vt, const float* st, float* dt) {
    float ds[8], dsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = umma::ex2(fmaf(st[i], kLog2e, -b2[i]));
      dt[i] = fmaf(w, gv[i], dt[i]);
      ds[i] = w * gv[i] * (vt[i] - P[i]);
      dsum += ds[i];
    }
    store8(dkp + (long long)t * d, dt);
    if (score_width == 1) {
      for (int o = 1; o < G; o <<= 1) dsum += __shfl_xor_sync(gmask, dsum, o);
      if (cgl == 0) atomicAdd(dsp + t, dsum);
    } else {
      store8(dsp + (long long)t * score_width + c0, ds);
    }
  };
#pragma unroll
  for (int k = 0; k < kSplitCache; ++k)
    if (k < n_my) {
      const float4 lo = *reinterpret_cast<const float4*>(&dk_s[k][0][tid][0]);
      const float4 hi = *reinterpret_cast<const float4*>(&dk_s[k][1][tid][0]);
      float dt[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      grad(ts + k * TS, vc[k], sc[k], dt);
    }
  for (int k = kSplitCache; k < n_my; ++k) {
    const int t = ts + k * TS;
    float vt[8], st[8], dt[8];
    load_token(kvp, scp, t, d, score_width, c0, vt, st);
    load8(dkp + (long long)t * d, dt);
    grad(t, vt, st, dt);
  }
}

namespace {
constexpr int kCompressThreads = 64;

template <typename T, int R>
void compress_fwd_t(const void* kv, long long kv_bs, const void* score, int score_width,
                    void* out, long long out_bs, int b, int sq, int d, int ratio, cudaStream_t s) {
  const int n_c = sq / ratio;
  if (R == 0 && ratio >= kSplitMinRatio) {
    const int G = split_slice_groups(d / 8);
    compress_split_kernel<T><<<dim3((unsigned)n_c, (unsigned)b, (unsigned)(d / 8 / G)),
                               kSplitThreads, 0, s>>>((const T*)kv, kv_bs, (const T*)score,
                                                      score_width, (T*)out, out_bs, sq, d,
                                                      ratio, G);
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
    const int G = split_slice_groups(d / 8);
    compress_bwd_split_kernel<T><<<dim3(nx, (unsigned)b, (unsigned)(d / 8 / G)), kSplitThreads, 0,
                                   s>>>((const T*)kv, kv_bs, (const T*)score, score_width, g, g_bs,
                                        dkv, dkv_bs, dscore, sq, d, ratio, n_c, G);
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
