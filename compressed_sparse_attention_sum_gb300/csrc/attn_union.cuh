// Slot set of a block of QB consecutive queries, shared by the tensor-core
// attention forward and backward.
//
// The block's queries see the window rows [t0 - W + 1, t_last] (one run of raw
// rows) and the compressed blocks any of them selected.  Per compressed block
// j the multiplicity of j in each query's index row is counted in shared
// memory, 16 bits per query packed four to a u64 (cnt[j][QB / 4]); the union
// is the ascending list of blocks with a non-zero count.  A repeated index is
// a repeated softmax term ("Add unfused SBHD compressed sparse attention",
// index_select gather), which the kernels apply as a log2(count) logit bias.
#pragma once
#include <cstdint>

namespace csa {

// CTA order: the work of a query block grows with its position (more visible
// compressed blocks), so the grid is issued heaviest first (longest job
// first), which keeps the last wave short.  Linear CTA id -> (batch, block).
__device__ __forceinline__ void heavy_first_block(int nblk, int* bi, int* xb) {
  const int b = (int)gridDim.x / nblk;
  const int id = blockIdx.x;
  *bi = id % b;
  *xb = nblk - 1 - id / b;
}

// Ascending compaction of the blocks below vmax with a non-zero count into
// ulist; returns the union size.  cnt must be complete and visible to all
// threads (after a barrier) on entry.
template <int QB, int kThreads>
__device__ __forceinline__ int union_compact(int vmax, const uint64_t* cnt, int* ulist, int* wsum,
                                             int* scal) {
  constexpr int NW = (QB + 3) / 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // ascending compaction: each thread scans a contiguous range of blocks
  const int per = (vmax + kThreads - 1) / kThreads;
  const int j0 = tid * per, j1 = min(vmax, j0 + per);
  int c = 0;
  for (int j = j0; j < j1; ++j) {
    bool any = false;
#pragma unroll
    for (int w = 0; w < NW; ++w) any |= cnt[j * NW + w] != 0ull;
    c += any;
  }
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  int pos = base + incl - c;
  for (int j = j0; j < j1; ++j) {
    bool any = false;
#pragma unroll
    for (int w = 0; w < NW; ++w) any |= cnt[j * NW + w] != 0ull;
    if (any) ulist[pos++] = j;
  }
  if (tid == kThreads - 1) scal[0] = base + incl;
  __syncthreads();
  return scal[0];
}

// Count multiplicities and build the ascending union list; returns its size.
// cnt must be zeroed and visible to all threads (after a barrier) on entry.
// idx == nullptr selects every visible block (dense mode).  The block's
// queries are t0 .. t0+QB-1 below t_end (t_end <= sq; sq is the row stride of
// idx).
template <int QB, int kThreads>
__device__ __forceinline__ int build_union(const int32_t* __restrict__ idx, int bi, int sq, int K,
                                           int t0, int t_end, int ratio, int n_c, uint64_t* cnt,
                                           int* ulist, int* wsum, int* scal) {
  constexpr int NW = (QB + 3) / 4;
  const int tid = threadIdx.x;
  const int t_last = min(t0 + QB, t_end) - 1;
  const int vmax = min((t_last + 1) / ratio, n_c);
  if (idx != nullptr) {
    for (int s0 = 0; s0 < K; s0 += kThreads) {
      const int s = s0 + tid;
      // all of this thread's loads are in flight before the first atomic
      int jv[QB];
#pragma unroll
      for (int q = 0; q < QB; ++q)
        jv[q] = (s < K && t0 + q < t_end) ? __ldg(idx + ((long long)bi * sq + t0 + q) * K + s)
                                          : -1;
#pragma unroll
      for (int q = 0; q < QB; ++q) {
        const int vis = min((t0 + q + 1) / ratio, n_c);
        if (jv[q] >= 0 && jv[q] < vis)
          atomicAdd(reinterpret_cast<unsigned long long*>(&cnt[jv[q] * NW + (q >> 2)]),
                    1ull << (16 * (q & 3)));
      }
    }
  } else {
    for (int q = 0; q < QB; ++q) {
      const int t = t0 + q;
      if (t >= t_end) break;
      const int vis = min((t + 1) / ratio, n_c);
      for (int j = tid; j < vis; j += kThreads)
        atomicAdd(reinterpret_cast<unsigned long long*>(&cnt[j * NW + (q >> 2)]),
                  1ull << (16 * (q & 3)));
    }
  }
  __syncthreads();
  return union_compact<QB, kThreads>(vmax, cnt, ulist, wsum, scal);
}

}  // namespace csa
