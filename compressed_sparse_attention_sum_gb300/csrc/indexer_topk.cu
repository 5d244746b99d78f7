// csa_indexer_topk: lightning-indexer scores and the exact causal top-k.
//
// Score: I[b,t,j] = sum_h w[b,t,h] * max(0, q_I[b,t,h,:] . k_I[b,j,:]) for
// j < vis(t) = (t+1)/ratio ("Add unfused SBHD compressed sparse attention",
// indexer block and causal compressed mask; "Refactor Deepseek v4 to use
// Attention Gym's Compressed Sparse Attention", indexer selectability).
// Selection: the K largest scores of each row, ties to the lower block index,
// emitted in ascending block order ("Add the min-memory DSA attention
// kernels": routing must be tie-exact with one full top-k; support sorted by
// position).
//
// This file holds the CUDA-core score kernel (fp32 inputs and any shape) and
// the per-row radix select that every score kernel feeds.  Scores of one
// chunk of query rows sit in a caller-provided fp32 workspace laid out
// [b][chunk rows][n_c]; only the visible prefix of each row is written and
// read, and a chunk is sized to stay resident in L2 between the two kernels.
#include <cuda_fp8.h>

#include <algorithm>

#include "csa_common.cuh"
#include "csa_kernels.h"

namespace csa {

// e4m3 code -> its exact fp32 value
__device__ __forceinline__ float to_f(__nv_fp8_e4m3 x) { return static_cast<float>(x); }

// ----------------------------------------------------------------------------
// CUDA-core score kernel: 64 query rows x 64 blocks per CTA, 256 threads,
// 4x4 outputs per thread; loops over the indexer heads.  With e4m3 codes
// (T = __nv_fp8_e4m3) the per-row scales enter as w[t,h] * q_scale[t,h] and a
// final factor k_scale[j] (both positive, so they commute with the ReLU).
// ----------------------------------------------------------------------------
constexpr int kSQ = 64;
constexpr int kSK = 64;

template <typename T>
__global__ void __launch_bounds__(256) indexer_scores_simt(
    const T* __restrict__ q_idx, const T* __restrict__ k_idx, const float* __restrict__ w,
    float* __restrict__ ws, int t0, int nt, int sq, int n_c, int H_I, int d_I, int ratio,
    const float* __restrict__ q_scale, const float* __restrict__ k_scale) {
  extern __shared__ float sm[];
  float* q_s = sm;                    // [d_I][kSQ]
  float* k_s = sm + d_I * kSQ;        // [d_I][kSK]
  float* w_s = k_s + d_I * kSK;       // [kSQ]
  const int bi = blockIdx.z;
  const int tq0 = t0 + blockIdx.y * kSQ;               // first query of the tile
  const int j0 = blockIdx.x * kSK;                     // first block of the tile
  const int tq_end = min(t0 + nt, tq0 + kSQ);          // exclusive
  if (tq0 >= tq_end) return;
  const int vis_max = min(tq_end / ratio, n_c);        // vis of the last query of the tile
  if (j0 >= vis_max) return;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;

  // keys of the tile (transposed)
  for (int e = tid; e < kSK * d_I; e += 256) {
    const int jj = e / d_I, c = e % d_I;
    const int j = j0 + jj;
    k_s[c * kSK + jj] = (j < n_c) ? to_f(k_idx[((long long)bi * n_c + j) * d_I + c]) : 0.f;
  }
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;

  for (int h = 0; h < H_I; ++h) {
    __syncthreads();
    for (int e = tid; e < kSQ * d_I; e += 256) {
      const int rr = e / d_I, c = e % d_I;
      const int t = tq0 + rr;
      q_s[c * kSQ + rr] =
          (t < tq_end) ? to_f(q_idx[(((long long)bi * sq + t) * H_I + h) * d_I + c]) : 0.f;
    }
    if (tid < kSQ) {
      const int t = tq0 + tid;
      const long long wi = ((long long)bi * sq + t) * H_I + h;
      w_s[tid] = (t < tq_end) ? (q_scale ? w[wi] * q_scale[wi] : w[wi]) : 0.f;
    }
    __syncthreads();
    float dot[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) dot[a][c] = 0.f;
    for (int c = 0; c < d_I; ++c) {
      const float4 qv = *reinterpret_cast<const float4*>(&q_s[c * kSQ + ty * 4]);
      const float4 kv = *reinterpret_cast<const float4*>(&k_s[c * kSK + tx * 4]);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
      const float ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) dot[a][cc] = fmaf(qa[a], ka[cc], dot[a][cc]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float wv = w_s[ty * 4 + a];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) acc[a][cc] = fmaf(wv, fmaxf(dot[a][cc], 0.f), acc[a][cc]);
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int t = tq0 + ty * 4 + a;
    if (t >= tq_end) continue;
    const int vis = min((t + 1) / ratio, n_c);
    float* dst = ws + ((long long)bi * nt + (t - t0)) * n_c;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int j = j0 + tx * 4 + cc;
      if (j < vis) dst[j] = k_scale ? acc[a][cc] * k_scale[(long long)bi * n_c + j] : acc[a][cc];
    }
  }
}

// ----------------------------------------------------------------------------
// Per-row exact top-K by 4-pass 8-bit radix select on order-preserving keys.
// One warp per query row.
//
// Candidates of row t: blocks j < vis(t); with per-token document ids (packed
// documents, "Refactor Deepseek v4 to use Attention Gym's Compressed Sparse
// Attention": block j belongs to doc[j*ratio] and is selectable by t only in
// t's document) only the blocks of t's document.  A non-candidate gets key 0,
// which no finite score maps to.  Rows with at most K candidates emit all of
// them, ascending, then -1.
// ----------------------------------------------------------------------------

// Emit every candidate (key != 0) of a row in ascending block order, then -1
// up to K.  keys_at(j) gives the key of block j.
template <typename KeyAt>
__device__ __forceinline__ void emit_all_candidates(int vis, int K, KeyAt keys_at,
                                                    const float* row, int32_t* oi, float* os) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  int out_pos = 0;
  for (int base = 0; base < vis; base += 32) {
    const int j = base + lane;
    const bool sel = j < vis && keys_at(j) != 0u;
    const unsigned selm = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int p = out_pos + __popc(selm & lt_mask);
      oi[p] = j;
      if (os) os[p] = row[j];
    }
    out_pos += __popc(selm);
  }
  for (int s = out_pos + lane; s < K; s += 32) {
    oi[s] = -1;
    if (os) os[s] = 0.f;
  }
}
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Row (b-major index into the chunk) of warp slot r0.  A row whose visible
// blocks number at most K selects all of them, so it needs no score: those
// rows come first, in ascending position, and run while the score grid is
// still busy (the select is its dependent launch); then the other rows, the
// most visible blocks first (the heavy rows start as soon as the scores are
// complete).  Batch elements are interleaved.  vis(t) <= K exactly for
// t <= (K+1)*ratio - 2 when n_c > K.
__device__ __forceinline__ int select_row(int r0, int b, int nt, int t0, int ratio, int n_c,
                                          int K) {
  const int ts = n_c <= K ? nt : min(max((K + 1) * ratio - 1 - t0, 0), nt);
  const int n_triv = b * ts;
  if (r0 < n_triv) return (r0 % b) * nt + r0 / b;
  const int r1 = r0 - n_triv;
  return (r1 % b) * nt + (nt - 1 - r1 / b);
}

__global__ void __launch_bounds__(256) topk_select_kernel(const float* __restrict__ ws,
                                                          int32_t* __restrict__ out_idx,
                                                          float* __restrict__ out_score, int t0,
                                                          int nt, int b, int sq, int n_c,
                                                          int ratio, int K,
                                                          const int32_t* __restrict__ doc) {
  extern __shared__ uint32_t smk[];
  const int warps = blockDim.x / 32;
  const int wid = threadIdx.x / 32, lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  uint32_t* keys = smk + (size_t)wid * (n_c + 256);
  int* hist = reinterpret_cast<int*>(keys + n_c);
  const int r0 = blockIdx.x * warps + wid;
  if (r0 >= b * nt) return;
  const int r = select_row(r0, b, nt, t0, ratio, n_c, K);
  const int bi = r / nt, t = t0 + r % nt;
  const int vis = min((t + 1) / ratio, n_c);
  const float* row = ws + (size_t)r * n_c;
  int32_t* oi = out_idx + ((size_t)bi * sq + t) * K;
  float* os = out_score ? out_score + ((size_t)bi * sq + t) * K : nullptr;
  // the score grid's output is read only where the selection depends on it
  // or the scores are returned (every thread of the warp decides alike)
  const bool scored = vis > K || os != nullptr;
  if (scored) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (doc == nullptr && vis <= K) {
    for (int s = lane; s < K; s += 32) {
      oi[s] = s < vis ? s : -1;
      if (os) os[s] = s < vis ? row[s] : 0.f;
    }
    return;
  }
  const int32_t* docb = doc ? doc + (size_t)bi * sq : nullptr;
  const int dt = docb ? docb[t] : 0;
  int ncand = 0;
  for (int j = lane; j < vis; j += 32) {
    const bool ok = docb == nullptr || __ldg(docb + (size_t)j * ratio) == dt;
    keys[j] = ok ? (scored ? order_key(row[j]) : 1u) : 0u;   // unscored: ncand <= vis <= K
    ncand += ok;
  }
  __syncwarp();
  ncand = __reduce_add_sync(FULL, ncand);
  if (ncand <= K) {
    emit_all_candidates(vis, K, [&](int j) { return keys[j]; }, row, oi, os);
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int need = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int j = lane; j < vis; j += 32) {
      const uint32_t u = keys[j];
      if (u != 0u && (u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
    }
    __syncwarp();
    // lane l owns bins 8*(31-l) .. 8*(31-l)+7, so lane 0 holds the highest bins
    int cnt[8];
    int tot = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cnt[i] = hist[8 * (31 - lane) + 7 - i];
      tot += cnt[i];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - tot;  // keys in bins above this lane's bins
    const bool mine = (excl < need) && (need <= incl);
    const unsigned bal = __ballot_sync(FULL, mine);
    const int src = __ffs(bal) - 1;
    int bin = 0, above = 0;
    if (mine) {
      int run = excl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (run + cnt[i] >= need) {
          bin = 8 * (31 - lane) + 7 - i;
          above = run;
          break;
        }
        run += cnt[i];
      }
    }
    bin = __shfl_sync(FULL, bin, src);
    above = __shfl_sync(FULL, above, src);
    need -= above;
    prefix |= (uint32_t)bin << shift;
    pmask |= 255u << shift;
    __syncwarp();
  }
  // threshold key = prefix: keep every key above it and the `need` lowest-index
  // keys equal to it, in ascending block order.
  int out_pos = 0, eq_seen = 0;
  for (int base = 0; base < vis; base += 32) {
    const int j = base + lane;
    const uint32_t u = (j < vis) ? keys[j] : 0u;
    const bool gt = u != 0u && u > prefix;
    const bool eq = u != 0u && u == prefix;
    const unsigned eqm = __ballot_sync(FULL, eq);
    const bool sel = gt || (eq && (eq_seen + __popc(eqm & lt_mask)) < need);
    const unsigned selm = __ballot_sync(FULL, sel);
    if (sel) {
      const int p = out_pos + __popc(selm & lt_mask);
      oi[p] = j;
      if (os) os[p] = row[j];
    }
    out_pos += __popc(selm);
    eq_seen += __popc(eqm);
  }
}

// Register-resident variant for rows of at most 32*PER candidates: lane l
// holds the keys of blocks l, l+32, ...  A pass whose chosen bin holds exactly
// the remaining count ends the search early: every key with the selected
// prefix is taken and no tie needs breaking.
template <int PER, bool DOC>
__global__ void __launch_bounds__(128) topk_select_reg_kernel(const float* __restrict__ ws,
                                                              int32_t* __restrict__ out_idx,
                                                              float* __restrict__ out_score,
                                                              int t0, int nt, int b, int sq,
                                                              int n_c, int ratio, int K,
                                                              const int32_t* __restrict__ doc) {
  __shared__ int hist_all[4][256];
  const int warps = blockDim.x / 32;
  const int wid = threadIdx.x / 32, lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  int* hist = hist_all[wid];
  const int r0 = blockIdx.x * warps + wid;
  if (r0 >= b * nt) return;
  const int r = select_row(r0, b, nt, t0, ratio, n_c, K);
  const int bi = r / nt, t = t0 + r % nt;
  const int vis = min((t + 1) / ratio, n_c);
  const float* row = ws + (size_t)r * n_c;
  int32_t* oi = out_idx + ((size_t)bi * sq + t) * K;
  float* os = out_score ? out_score + ((size_t)bi * sq + t) * K : nullptr;
  // the score grid's output is read only where the selection depends on it
  // or the scores are returned (every thread of the warp decides alike); with
  // document ids that is known only from the candidates' count, which needs
  // the ids alone (an input, not the score grid's output)
  bool scored = vis > K || os != nullptr;
  if (!DOC && scored) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!DOC && vis <= K) {
    for (int s = lane; s < K; s += 32) {
      oi[s] = s < vis ? s : -1;
      if (os) os[s] = s < vis ? row[s] : 0.f;
    }
    return;
  }
  const int32_t* docb = DOC ? doc + (size_t)bi * sq : nullptr;
  const int dt = DOC ? docb[t] : 0;
  uint32_t key[PER];
  int ncand = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int j = lane + 32 * i;
    const bool ok = j < vis && (!DOC || __ldg(docb + (size_t)j * ratio) == dt);
    key[i] = ok ? 1u : 0u;                             // 0: not a candidate
    ncand += ok;
  }
  if (DOC) {
    ncand = __reduce_add_sync(FULL, ncand);
    scored = ncand > K || os != nullptr;
    if (scored) asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  if (scored) {
    // unscored rows (ncand <= K) only mark their candidates
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (key[i] != 0u) key[i] = order_key(row[lane + 32 * i]);
  }
  if (DOC && ncand <= K) {
    // blocks l, l+32, ...: fetch the key of block j from its owner lane
    int out_pos = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (32 * i >= vis) break;
      const int j = lane + 32 * i;
      const bool sel = key[i] != 0u;
      const unsigned selm = __ballot_sync(FULL, sel);
      if (sel) {
        const int p = out_pos + __popc(selm & lt_mask);
        oi[p] = j;
        if (os) os[p] = row[j];
      }
      out_pos += __popc(selm);
    }
    for (int s2 = out_pos + lane; s2 < K; s2 += 32) {
      oi[s2] = -1;
      if (os) os[s2] = 0.f;
    }
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int need = K;
  bool exact = false;                                  // true: a bin matched `need` exactly
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int j = lane + 32 * i;
      const bool cand = DOC ? key[i] != 0u : j < vis;
      if (cand && (key[i] & pmask) == prefix) atomicAdd(&hist[(key[i] >> shift) & 255u], 1);
    }
    __syncwarp();
    int cnt[8];
    int tot = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cnt[i] = hist[8 * (31 - lane) + 7 - i];
      tot += cnt[i];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - tot;
    const bool mine = (excl < need) && (need <= incl);
    const int src = __ffs(__ballot_sync(FULL, mine)) - 1;
    int bin = 0, above = 0, inbin = 0;
    if (mine) {
      int run = excl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (run + cnt[i] >= need) {
          bin = 8 * (31 - lane) + 7 - i;
          above = run;
          inbin = cnt[i];
          break;
        }
        run += cnt[i];
      }
    }
    bin = __shfl_sync(FULL, bin, src);
    above = __shfl_sync(FULL, above, src);
    inbin = __shfl_sync(FULL, inbin, src);
    need -= above;
    prefix |= (uint32_t)bin << shift;
    pmask |= 255u << shift;
    __syncwarp();
    if (inbin == need) {
      exact = true;
      break;
    }
  }
  int out_pos = 0, eq_seen = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int j = lane + 32 * i;
    if (32 * i >= vis) break;
    const uint32_t u = key[i];
    const bool valid = DOC ? u != 0u : j < vis;
    bool sel;
    unsigned eqm = 0u;
    if (exact) {
      sel = valid && (u & pmask) >= prefix;
    } else {
      const bool eq = valid && u == prefix;
      eqm = __ballot_sync(FULL, eq);
      sel = (valid && u > prefix) || (eq && (eq_seen + __popc(eqm & lt_mask)) < need);
    }
    const unsigned selm = __ballot_sync(FULL, sel);
    if (sel) {
      const int p = out_pos + __popc(selm & lt_mask);
      oi[p] = j;
      if (os) os[p] = row[j];
    }
    out_pos += __popc(selm);
    eq_seen += __popc(eqm);
  }
}

// Rows without document ids, a CTA of four warps per row that has more than
// K visible blocks (a warp per row only for the rows that take all their
// blocks): thread i holds the keys of blocks i, i+128, ..., the radix passes
// count into a CTA-shared histogram (two, alternating, so that one is cleared
// while the other is scanned), and the row is written in ascending block order
// from per-warp counts.  A row's selection then takes a quarter of the
// dependent steps of one warp walking all its keys, which matters because the
// rows that depend on the scores all start when the score grid completes.
// CTAs [0, light) take four rows that keep all their blocks each (ascending
// positions, no wait unless scores are returned), the others one row with
// more than K blocks each, heaviest first, batch elements interleaved.
template <int PH>
__global__ void __launch_bounds__(128) topk_select_cta_kernel(const float* __restrict__ ws,
                                                              int32_t* __restrict__ out_idx,
                                                              float* __restrict__ out_score,
                                                              int t0, int nt, int b, int sq,
                                                              int n_c, int ratio, int K) {
  __shared__ int hist[2][256];
  __shared__ int res[2][4];
  __shared__ int wcount[2][4][PH];           // per (warp, key index): ties, then selected
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const unsigned FULL = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int ts = n_c <= K ? nt : min(max((K + 1) * ratio - 1 - t0, 0), nt);
  const int n_light = b * ts, light_ctas = (n_light + 3) / 4;
  if ((int)blockIdx.x < light_ctas) {
    const int r0 = blockIdx.x * 4 + wid;
    if (r0 >= n_light) return;
    const int r = (r0 % b) * nt + r0 / b;
    const int bi = r / nt, t = t0 + r % nt;
    const int vis = min((t + 1) / ratio, n_c);
    const float* row = ws + (size_t)r * n_c;
    int32_t* oi = out_idx + ((size_t)bi * sq + t) * K;
    float* os = out_score ? out_score + ((size_t)bi * sq + t) * K : nullptr;
    if (os) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int s2 = lane; s2 < K; s2 += 32) {
      oi[s2] = s2 < vis ? s2 : -1;
      if (os) os[s2] = s2 < vis ? row[s2] : 0.f;
    }
    return;
  }
  const int h = blockIdx.x - light_ctas;
  const int r = (h % b) * nt + (nt - 1 - h / b);
  const int bi = r / nt, t = t0 + r % nt;
  const int vis = min((t + 1) / ratio, n_c);         // > K
  const float* row = ws + (size_t)r * n_c;
  int32_t* oi = out_idx + ((size_t)bi * sq + t) * K;
  float* os = out_score ? out_score + ((size_t)bi * sq + t) * K : nullptr;
  for (int e = tid; e < 512; e += 128) (&hist[0][0])[e] = 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint32_t key[PH];
#pragma unroll
  for (int i = 0; i < PH; ++i) {
    const int j = tid + 128 * i;
    key[i] = j < vis ? order_key(row[j]) : 0u;
  }
  __syncthreads();
  uint32_t prefix = 0, pmask = 0;
  int need = K;
  bool exact = false;
  for (int shift = 24, ps = 0; shift >= 0; shift -= 8, ps ^= 1) {
    int* H = hist[ps];
#pragma unroll
    for (int i = 0; i < PH; ++i) {
      const int j = tid + 128 * i;
      if (j < vis && (key[i] & pmask) == prefix) atomicAdd(&H[(key[i] >> shift) & 255u], 1);
    }
    __syncthreads();
    if (wid == 0) {
      // bins in descending order: lane l scans bins 8(31-l)+7 .. 8(31-l)
      int cnt[8];
      int tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = H[8 * (31 - lane) + 7 - i];
        tot += cnt[i];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = incl - tot;
      if (excl < need && need <= incl) {              // exactly one lane
        int run = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run + cnt[i] >= need) {
            res[ps][0] = 8 * (31 - lane) + 7 - i;
            res[ps][1] = run;
            res[ps][2] = cnt[i];
            break;
          }
          run += cnt[i];
        }
      }
    } else if (wid == 1) {
      // the other histogram (last read by the previous pass's scan) for the next pass
      for (int e = lane; e < 256; e += 32) hist[ps ^ 1][e] = 0;
    }
    __syncthreads();
    const int bin = res[ps][0], above = res[ps][1], inbin = res[ps][2];
    need -= above;
    prefix |= (uint32_t)bin << shift;
    pmask |= 255u << shift;
    if (inbin == need) {
      exact = true;
      break;
    }
  }
  // selection in ascending block order j = 128 i + 32 wid + lane
  bool sel[PH];
  if (exact) {
#pragma unroll
    for (int i = 0; i < PH; ++i)
      sel[i] = tid + 128 * i < vis && (key[i] & pmask) >= prefix;
  } else {
    // the threshold key's `need` lowest-index copies are taken
    unsigned eqm[PH];
#pragma unroll
    for (int i = 0; i < PH; ++i) {
      const bool eq = tid + 128 * i < vis && key[i] == prefix;
      eqm[i] = __ballot_sync(FULL, eq);
      if (lane == 0) wcount[0][wid][i] = __popc(eqm[i]);
    }
    __syncthreads();
    int run = 0;
#pragma unroll
    for (int i = 0; i < PH; ++i) {
      int before = 0, tot = 0;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int c = wcount[0][w][i];
        before += w < wid ? c : 0;
        tot += c;
      }
      const bool valid = tid + 128 * i < vis;
      const bool eq = (eqm[i] >> lane) & 1u;
      sel[i] = (valid && key[i] > prefix) || (eq && run + before + __popc(eqm[i] & lt_mask) < need);
      run += tot;
    }
  }
  unsigned selm[PH];
#pragma unroll
  for (int i = 0; i < PH; ++i) {
    selm[i] = __ballot_sync(FULL, sel[i]);
    if (lane == 0) wcount[1][wid][i] = __popc(selm[i]);
  }
  __syncthreads();
  int run = 0;
#pragma unroll
  for (int i = 0; i < PH; ++i) {
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int c = wcount[1][w][i];
      before += w < wid ? c : 0;
      tot += c;
    }
    const int pos = run + before + __popc(selm[i] & lt_mask);
    if (sel[i] && pos < K) {
      const int j = tid + 128 * i;
      oi[pos] = j;
      if (os) os[pos] = row[j];
    }
    run += tot;
  }
}

cudaError_t launch_indexer_scores_simt(const void* q_idx, const void* k_idx, const float* w,
                                       float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                       int d_I, int ratio, bool bf16, cudaStream_t s) {
  dim3 grid((unsigned)((n_c + kSK - 1) / kSK), (unsigned)((nt + kSQ - 1) / kSQ), (unsigned)b);
  const size_t smem = (size_t)(d_I * (kSQ + kSK) + kSQ) * sizeof(float);
  if (bf16) {
    auto k = indexer_scores_simt<__nv_bfloat16>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<grid, 256, smem, s>>>((const __nv_bfloat16*)q_idx, (const __nv_bfloat16*)k_idx, w, ws, t0,
                              nt, sq, n_c, H_I, d_I, ratio, nullptr, nullptr);
    count_launches(1);
  } else {
    auto k = indexer_scores_simt<float>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<grid, 256, smem, s>>>((const float*)q_idx, (const float*)k_idx, w, ws, t0, nt, sq, n_c,
                              H_I, d_I, ratio, nullptr, nullptr);
    count_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_indexer_scores_simt_fp8(const uint8_t* q8, const float* q_scale,
                                           const uint8_t* k8, const float* k_scale,
                                           const float* w, float* ws, int t0, int nt, int b,
                                           int sq, int n_c, int H_I, int d_I, int ratio,
                                           cudaStream_t s) {
  dim3 grid((unsigned)((n_c + kSK - 1) / kSK), (unsigned)((nt + kSQ - 1) / kSQ), (unsigned)b);
  const size_t smem = (size_t)(d_I * (kSQ + kSK) + kSQ) * sizeof(float);
  auto k = indexer_scores_simt<__nv_fp8_e4m3>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k<<<grid, 256, smem, s>>>((const __nv_fp8_e4m3*)q8, (const __nv_fp8_e4m3*)k8, w, ws, t0, nt,
                            sq, n_c, H_I, d_I, ratio, q_scale, k_scale);
  count_launches(1);
  return cudaGetLastError();
}

// Packed documents must start on multiples of the ratio, so that no pooled
// block mixes two documents ("Refactor Deepseek v4 to use Attention Gym's
// Compressed Sparse Attention": packing pads every document to a multiple of
// the compress ratio).  A document id that changes inside a block records
// CSA_ERR_DEVICE_CHECK at kSiteDocBoundary; the results are still computed
// under the rule that a block belongs to the document of its first token.
__global__ void doc_boundary_check_kernel(const int32_t* __restrict__ doc, long long n, int sq,
                                          int ratio, int* __restrict__ status) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i % sq);
    if (t % ratio != 0 && __ldg(doc + i) != __ldg(doc + i - 1)) {
      set_status(status, kDevCheck, kSiteDocBoundary);
      return;
    }
  }
}

cudaError_t launch_doc_boundary_check(const int32_t* doc, int b, int sq, int ratio, int* status,
                                      cudaStream_t s) {
  const long long n = (long long)b * sq;
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const unsigned grid = (unsigned)(want < 1024 ? (want < 1 ? 1 : want) : 1024);
  doc_boundary_check_kernel<<<grid, threads, 0, s>>>(doc, n, sq, ratio, status);
  count_launches(1);
  return cudaGetLastError();
}

// Launch a kernel that may be scheduled before the preceding kernel on the
// stream has completed (programmatic dependent launch): the kernel waits for
// it with griddepcontrol.wait before reading its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_topk_select(const float* ws, int32_t* topk_idx, float* topk_score, int t0,
                               int nt, int b, int sq, int n_c, int ratio, int K, cudaStream_t s,
                               const int32_t* doc) {
  const int rows = b * nt;
  if (doc == nullptr && n_c <= 2048) {
    const int ts = n_c <= K ? nt : std::min(std::max((K + 1) * ratio - 1 - t0, 0), nt);
    const unsigned grid = (unsigned)((b * ts + 3) / 4 + b * (nt - ts));
#define CSA_SELC(P)                                                                           \
  {                                                                                           \
    cudaError_t e_ = launch_dependent(topk_select_cta_kernel<P>, grid, 128, 0, s, ws, topk_idx,\
                                      topk_score, t0, nt, b, sq, n_c, ratio, K);              \
    if (e_ != cudaSuccess) return e_;                                                         \
    count_launches(1);                                                                        \
  }
    if (n_c <= 256) { CSA_SELC(2) }
    else if (n_c <= 512) { CSA_SELC(4) }
    else if (n_c <= 1024) { CSA_SELC(8) }
    else { CSA_SELC(16) }
#undef CSA_SELC
    return cudaGetLastError();
  }
  if (n_c <= 2048) {
    const unsigned grid = (unsigned)((rows + 3) / 4);   // 4 rows (warps) per CTA
#define CSA_SEL(P)                                                                            \
  {                                                                                           \
    cudaError_t e_ = doc ? launch_dependent(topk_select_reg_kernel<P, true>, grid, 128, 0, s, \
                                            ws, topk_idx, topk_score, t0, nt, b, sq, n_c,     \
                                            ratio, K, doc)                                    \
                         : launch_dependent(topk_select_reg_kernel<P, false>, grid, 128, 0, s,\
                                            ws, topk_idx, topk_score, t0, nt, b, sq, n_c,     \
                                            ratio, K, (const int32_t*)nullptr);               \
    if (e_ != cudaSuccess) return e_;                                                         \
    count_launches(1);                                                                        \
  }
    if (n_c <= 256) { CSA_SEL(8) }
    else if (n_c <= 512) { CSA_SEL(16) }
    else if (n_c <= 1024) { CSA_SEL(32) }
    else { CSA_SEL(64) }
#undef CSA_SEL
    return cudaGetLastError();
  }
  const size_t per_warp = (size_t)(n_c + 256) * sizeof(uint32_t);
  int warps = (int)((200 * 1024) / per_warp);
  warps = warps < 1 ? 1 : (warps > 8 ? 8 : warps);
  const size_t smem = per_warp * warps;
  dim3 grid((unsigned)((rows + warps - 1) / warps));
  cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_dependent(topk_select_kernel, grid, warps * 32, smem, s, ws, topk_idx,
                                   topk_score, t0, nt, b, sq, n_c, ratio, K, doc);
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
