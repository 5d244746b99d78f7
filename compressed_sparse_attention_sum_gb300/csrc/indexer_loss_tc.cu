// The indexer's distillation loss and its gradients on the 5th-generation
// tensor cores (tcgen05 + TMEM): bf16, d_I = 128, H_I in {32, 64}.
//
// Semantics as csa_indexer_loss ("Refactor Deepseek v4 to use Attention Gym's
// Compressed Sparse Attention": lightning indexer, a second pass over the
// selected entries only; "Add unfused SBHD compressed sparse attention",
// review of the teacher normalization): per query t and valid slot s,
//   I[s] = sum_h w[t,h] max(0, q_I[t,h] . k_I[j_s]),  p = softmax(I),
//   loss = sum_s target[s] (log target[s] - log p[s]),  dI = p sum(target) - target,
//   G[h,s] = dI[s] w[t,h] [q_I[t,h] . k_I[j_s] > 0],
//   dq_I[t,h] = sum_s G[h,s] k_I[j_s],  dw[t,h] = sum_s dI[s] max(0, q_I[t,h] . k_I[j_s]),
//   dk_I[j] += sum over (t, s: j_s = j) sum_h G[h,s] q_I[t,h].
//
// A CTA owns QB = 128 / H_I consecutive queries (128 (query, head) rows) and
// walks the ascending union of the blocks they selected, 128 at a time (the
// selections of neighbouring queries overlap, so one gathered k_I tile and
// one dk_I reduction serve all QB queries).  A query sees a union entry u
// through its multiplicity c(u) (0 = not selected; a repeated entry is c
// softmax terms), and its target mass T(u) is the sum of the targets of its
// slots holding u.  Products, transposed so that the union entry is the TMEM
// lane (M = 128) and the 128 rows are the N dimension:
//   X^T [slots, rows]  = K [slots, d] . Q^T            (dots; K-major A and B)
//   dQ^T [d, rows]    += K^T [d, slots] . G^T           (A = K and B = G MN-major)
//   dK^T [d, slots]    = Q^T [d, rows] . G [rows, slots] (A = Q MN-major, B = G K-major)
// G carries bf16 hi + lo parts (about 16 significant bits).  Pass A forms X^T
// and I for every union entry (two 128-column X^T buffers in TMEM) and keeps
// the sign of every dot, one bit per (entry, row), in TMEM; one CTA-wide
// softmax per query follows.  Pass B needs no dots: G comes from the sign
// bits, dI and w; dQ^T accumulates in TMEM and dK^T alternates between the
// two former X^T buffers, so a tile's dK^T columns are added into dk_I (fp32
// vector reductions, four block rows of 128 bytes per warp instruction) while
// the tensor core forms the next tile's products.  dw needs the dots' values:
//   dw[t,h] = sum_s dI[s] [dot > 0] (q_I[t,h] . k_I[j_s]) = q_I[t,h] . dq_I[t,h] / w[t,h],
// formed from dQ^T and the Q rows at the end (a row whose |w| is below 2^-60
// takes G with weight 1 instead, its dq_I scaled by w afterwards, and its Q
// row zeroed for the dK^T product).
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"
#include "attn_union.cuh"

#include <cudaTypedefs.h>

namespace csa {
namespace ilt {

using namespace csa::umma;

constexpr int kDI = 128;
constexpr int kRows = 128;                      // (query, head) rows: QB x H_I
constexpr int kSlots = 128;                     // union entries per tile
constexpr int kThreads = 512;                   // 16 warps: TMEM lane quarter x column quarter
constexpr uint32_t kTmemCols = 512;
// TMEM columns: pass A's X^T buffers (pass B: dK^T buffers) of 128 at 0 and
// 128, dQ^T at 256, the sign bits at 384 (four columns per tile: at most 32
// tiles, i.e. n_c <= 4096)
constexpr uint32_t kColDQ = 256, kColMask = 384;
constexpr float kTinyW = 8.673617379884035e-19f;   // 2^-60
constexpr uint32_t kBlk = 128 * 128;            // 16 KB: 128 lines of 128 B

struct Layout {
  static constexpr uint32_t Q = 0;              // [2][128 rows][128 B]
  static constexpr uint32_t KV = 2 * kBlk;      // two buffers of [2][128 slots][128 B]
  static constexpr uint32_t GH = 6 * kBlk;      // G hi [2][128 slots][128 B]
  static constexpr uint32_t GL = 8 * kBlk;      // G lo [2][128 slots][128 B]
  static constexpr uint32_t BARS = 10 * kBlk;   // q, x[4], s[2], dq, dk
  static constexpr uint32_t TSLOT = BARS + 9 * 8;
  static constexpr uint32_t SCAL = TSLOT + 8;   // [16] ints
  static constexpr uint32_t W = SCAL + 64;      // [128] floats: w of each row (0: no query)
  static constexpr uint32_t RED = W + 512;      // [4][128] floats
  static constexpr uint32_t QST = RED + 2048;   // [4][8] floats: per-query statistics
  static constexpr uint32_t SCR = QST + 128;    // [16][12] floats: block reductions
  static constexpr uint32_t WSUM = SCR + 768;   // [16] ints
  static constexpr uint32_t WG = WSUM + 64;     // [128] floats: G's weight per row
  static constexpr uint32_t DYN = WG + 512;     // cnt, ulist, I/dI, T
};
// per-query statistics in QST[q * 8 + k]
constexpr int kStS = 0, kStA = 1, kStLoss = 2, kStN = 3;

__device__ __forceinline__ uint32_t sw_off(int r, int ch) {
  return (uint32_t)((ch >> 3) * kBlk + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async_16_zf(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// bf16 hi and bf16 residual of 8 values, to two 16-byte chunks
__device__ __forceinline__ void store_hi_lo8(unsigned char* X, unsigned char* Y, uint32_t off,
                                             const float (&v)[8]) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
    hi[e] = *reinterpret_cast<const uint32_t*>(&h);
    lo[e] = *reinterpret_cast<const uint32_t*>(&l);
  }
  *reinterpret_cast<uint4*>(X + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(Y + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// CTA-wide sum (kMax: maximum) of N values per thread; every thread gets the
// results.  scr holds [16][N] floats.
template <int N, bool kMax>
__device__ __forceinline__ void block_reduce(float (&v)[N], float* scr) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    v[q] = kMax ? warp_max(v[q]) : warp_sum(v[q]);
    if (lane == 0) scr[warp * N + q] = v[q];
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < N; ++q) {
    float a = kMax ? -INFINITY : 0.f;
    for (int w = 0; w < kThreads / 32; ++w) a = kMax ? fmaxf(a, scr[w * N + q]) : a + scr[w * N + q];
    v[q] = a;
  }
  __syncthreads();
}

// Transposing butterfly over the 32 lanes: v[c] (c < 16) holds this lane's
// value of column c; afterwards lanes l and l + 16 hold the sum over all 32
// lanes of column l % 16.
__device__ __forceinline__ float lane_transpose_sum16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 8, n = 8; off >= 1; off >>= 1, n >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = up ? v[i] : v[i + n];
      const float keep = up ? v[i + n] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// 4x4 transposes within each quad of lanes: on entry lane 4a+b holds in x[j]
// the element (row b, column j) of its quad's block, on return in x[i] the
// element (row i, column b).  Two exchange steps (partner lane ^ 2, then
// ^ 1), each moving the elements whose row and column differ in that bit.
__device__ __forceinline__ void quad_transpose4(float (&x)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 2; s >= 1; s >>= 1) {
    const bool hi = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j & s) continue;
      const float send = hi ? x[j] : x[j ^ s];
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      if (hi) x[j] = recv;
      else x[j ^ s] = recv;
    }
  }
}

template <int QB>
__global__ void __launch_bounds__(kThreads, 1) indexer_loss_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __nv_bfloat16* __restrict__ q_I,
    const __nv_bfloat16* __restrict__ k_I, const float* __restrict__ w,
    const int32_t* __restrict__ idx,
    const float* __restrict__ target, float* __restrict__ loss, float* __restrict__ dq_I,
    float* __restrict__ dk_I, float* __restrict__ dw, int sq, int n_c, int ratio, int K,
    int* __restrict__ status) {
  constexpr int H_I = kRows / QB;
  constexpr int NW = (QB + 3) / 4;
  constexpr int GPQ = H_I / 32;                 // column groups (of 32 rows) per query
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + Layout::BARS);
  uint64_t* bar_x = bar_q + 1;                  // [2] pass-A X^T buffers
  uint64_t* bar_dk = bar_q + 3;                 // pass-B dQ^T and dK^T MMAs of a tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::TSLOT);
  int* scal = reinterpret_cast<int*>(sm + Layout::SCAL);
  float* wr = reinterpret_cast<float*>(sm + Layout::W);
  float* wg = reinterpret_cast<float*>(sm + Layout::WG);
  float* red = reinterpret_cast<float*>(sm + Layout::RED);
  float* qst = reinterpret_cast<float*>(sm + Layout::QST);
  float* scr = reinterpret_cast<float*>(sm + Layout::SCR);
  int* wsum = reinterpret_cast<int*>(sm + Layout::WSUM);
  uint64_t* cnt = reinterpret_cast<uint64_t*>(sm + Layout::DYN);   // [n_c][NW]
  int* ulist = reinterpret_cast<int*>(cnt + (size_t)n_c * NW);     // [n_c]
  float* Iu = reinterpret_cast<float*>(ulist + n_c);               // [QB][n_c]: I, then dI
  float* Tu = Iu + (size_t)QB * n_c;                               // [QB][n_c]: target mass per block
  unsigned char* GH = sm + Layout::GH;
  unsigned char* GL = sm + Layout::GL;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bi, xb;
  heavy_first_block((sq + QB - 1) / QB, &bi, &xb);
  const int t0 = xb * QB;
  const __nv_bfloat16* k_b = k_I + (long long)bi * n_c * kDI;
  float* dk_b = dk_I + (long long)bi * n_c * kDI;

  // ---- set-up: barriers, TMEM, Q tile, head weights ----------------------------
  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&bar_x[i], 1);
    mbar_init(bar_dk, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  for (int e = tid; e < n_c * NW; e += kThreads) cnt[e] = 0ull;
  for (int e = tid; e < QB * n_c; e += kThreads) Tu[e] = 0.f;
  if (tid < kRows) {
    const int q = tid / H_I, t = t0 + q;
    wr[tid] = t < sq ? w[((long long)bi * sq + t) * H_I + tid % H_I] : 0.f;
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    mbar_expect_tx(bar_q, 2 * kBlk);
    const int row0 = (bi * sq + t0) * H_I;
    tma_load_2d(sm + Layout::Q, &tmap_q, bar_q, 0, row0);
    tma_load_2d(sm + Layout::Q + kBlk, &tmap_q, bar_q, 64, row0);
  }

  // ---- union of the selected blocks, with each query's target mass per block ------
  // (multiplicities in cnt, target mass in Tu[q][j]; sum(target), sum t log t
  // and the number of valid slots per query in st)
  float st[3 * QB];
#pragma unroll
  for (int i = 0; i < 3 * QB; ++i) st[i] = 0.f;
  for (int s0 = 0; s0 < K; s0 += kThreads) {
    const int s = s0 + tid;
    int jv[QB];
    float tv[QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) {               // all loads in flight before the atomics
      const bool in = s < K && t0 + q < sq;
      const long long o = ((long long)bi * sq + t0 + q) * K + s;
      jv[q] = in ? __ldg(idx + o) : -1;
      tv[q] = in ? __ldg(target + o) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const int vis = min((t0 + q + 1) / ratio, n_c);
      if (jv[q] >= 0 && jv[q] < vis) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&cnt[jv[q] * NW + (q >> 2)]),
                  1ull << (16 * (q & 3)));
        atomicAdd(&Tu[q * n_c + jv[q]], tv[q]);
        st[q] += tv[q];
        if (tv[q] > 0.f) st[QB + q] += tv[q] * logf(tv[q]);
        st[2 * QB + q] += 1.f;
      }
    }
  }
  __syncthreads();
  const int n_u = union_compact<QB, kThreads>(min((min(t0 + QB, sq)) / ratio, n_c), cnt, ulist,
                                              wsum, scal);
  const int ntiles = (n_u + kSlots - 1) / kSlots;
  const int qd = warp & 3, cg = warp >> 2;          // lane quarter, column group (32 rows)
  const int r = qd * 32 + lane;                     // TMEM lane: union slot (X^T) or d (dQ^T, dK^T)
  const int myq = (cg * 32) / H_I;                  // the query of this thread's 32 rows
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;

  // gather union tile it into KV buffer `buf` (four in pass A, where the G
  // area is still free; two in pass B); padding slots are zeros
  auto stage = [&](int it, int buf) {
    const int sbase = it * kSlots;
    unsigned char* dst = sm + Layout::KV + buf * 2 * kBlk;
    for (int c = tid; c < kSlots * 16; c += kThreads) {
      const int rr = c >> 4, ch = c & 15;
      const bool pad = sbase + rr >= n_u;
      const __nv_bfloat16* src = k_b + (pad ? 0ll : (long long)ulist[sbase + rr] * kDI) + ch * 8;
      cp_async_16_zf(dst + sw_off(rr, ch), src, pad ? 0u : 16u);
    }
    cp_commit();
  };
  // X^T of the tile in KV buffer `buf` into the 128 TMEM columns at `col`
  auto issue_x = [&](int buf, uint32_t col, uint64_t* bar) {
    constexpr uint32_t idesc = idesc_bf16_f32_major(kSlots, kRows, 0, 0);
    const uint32_t ka = smem_addr(sm + Layout::KV + buf * 2 * kBlk);
    const uint32_t qa = smem_addr(sm + Layout::Q);
#pragma unroll
    for (int k = 0; k < kDI / 16; ++k) {
      const uint32_t off = (k >> 2) * kBlk + (k & 3) * 32;
      mma_bf16_ss(tmem + col, sw128_desc(ka + off), sw128_desc(qa + off), idesc,
                  k > 0 ? 1u : 0u);
    }
    mma_commit(bar);
  };

  // the first three tiles of pass A stream in while the statistics are reduced
  for (int i = 0; i < 3 && i < ntiles; ++i) stage(i, i);

  {
    block_reduce<3 * QB, false>(st, scr);
    if (tid == 0) {
#pragma unroll
      for (int q = 0; q < QB; ++q) {
        qst[q * 8 + kStS] = st[q];
        qst[q * 8 + kStA] = st[QB + q];
        qst[q * 8 + kStN] = st[2 * QB + q];
        qst[q * 8 + kStLoss] = st[QB + q];           // minus sum T log p, added below
      }
    }
  }
  bool ok = __syncthreads_and(mbar_wait(bar_q, 0));
  int site = ok ? 0 : kSiteLossQ;

  auto mult = [&](int q, int u) -> float {
    return (float)((uint32_t)(cnt[ulist[u] * NW + (q >> 2)] >> (16 * (q & 3))) & 0xFFFFu);
  };

  // ---- pass A: I for every union entry, with a running (max, sum) per query --------
  // Four KV buffers (tile it+3 is gathered while tile it is reduced) and two
  // X^T buffers (tile it+1's product runs while tile it is reduced); each
  // thread keeps the signs of its 32 dots of the tile in one TMEM word.
  float m_run[QB], z_run[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    m_run[q] = -INFINITY;
    z_run[q] = 0.f;
  }
  if (ok && ntiles > 0) {
    if (ntiles > 2) cp_wait<2>();
    else if (ntiles > 1) cp_wait<1>();
    else cp_wait<0>();
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0) {
      fence_after();
      issue_x(0, 0, &bar_x[0]);
    }
  }
  for (int it = 0; it < ntiles && ok; ++it) {
    if (it + 1 < ntiles) {
      // tile it+1 has arrived (tile it+2, if any, may still be in flight)
      if (it + 2 < ntiles) cp_wait<1>();
      else cp_wait<0>();
      fence_proxy_async_smem();
      fence_before();
      __syncthreads();
      if (tid == 0) {
        fence_after();
        issue_x((it + 1) & 3, ((it + 1) & 1) * 128, &bar_x[(it + 1) & 1]);
      }
    } else {
      __syncthreads();     // the previous tile's combine has read `red`
    }
    // per-warp wait: a warp scores its columns as soon as X^T is there, not
    // after the issuing thread has handed the next tile's product over (the
    // barrier below carries a failed wait to every thread)
    ok = __all_sync(0xffffffffu, mbar_wait(&bar_x[it & 1], (it >> 1) & 1));
    if (ok) {
      fence_after();
      uint32_t v[32];
      tmem_ld32_wait(tmem + lane_base + (it & 1) * 128 + cg * 32, v);
      const float4* w4 = reinterpret_cast<const float4*>(wr + cg * 32);
      float part = 0.f;
      uint32_t signs = 0u;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 wv = w4[c4];
        const float x0 = __uint_as_float(v[4 * c4]), x1 = __uint_as_float(v[4 * c4 + 1]);
        const float x2 = __uint_as_float(v[4 * c4 + 2]), x3 = __uint_as_float(v[4 * c4 + 3]);
        part = fmaf(wv.x, fmaxf(x0, 0.f), part);
        part = fmaf(wv.y, fmaxf(x1, 0.f), part);
        part = fmaf(wv.z, fmaxf(x2, 0.f), part);
        part = fmaf(wv.w, fmaxf(x3, 0.f), part);
        signs |= ((x0 > 0.f ? 1u : 0u) | (x1 > 0.f ? 2u : 0u) | (x2 > 0.f ? 4u : 0u) |
                  (x3 > 0.f ? 8u : 0u)) << (4 * c4);
      }
      red[cg * kRows + r] = part;
      tmem_st1(tmem + lane_base + kColMask + it * 4 + cg, signs);
    }
    fence_before();
    ok = __syncthreads_and(ok);
    if (!ok) { site = kSiteLossX; break; }
    if (tid < kSlots) {
      const int u = it * kSlots + tid;
      if (u < n_u) {
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          float s = 0.f;
#pragma unroll
          for (int g = 0; g < GPQ; ++g) s += red[(q * GPQ + g) * kRows + tid];
          Iu[q * n_c + u] = s;
          const float c = mult(q, u);
          if (c > 0.f) {                             // online softmax mass of this lane
            if (s > m_run[q]) {
              z_run[q] = z_run[q] * expf(m_run[q] - s) + c;
              m_run[q] = s;
            } else {
              z_run[q] += c * expf(s - m_run[q]);
            }
          }
        }
      }
    }
    // KV buffer (it+3) & 3 last held tile it-1, whose X^T has completed
    if (it + 3 < ntiles) stage(it + 3, (it + 3) & 3);
  }

  // ---- softmax per query: the lanes' (max, mass) joined; loss and dI ----------------
  __syncthreads();
  if (ok) {
    float m[QB], z[QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) m[q] = m_run[q];
    block_reduce<QB, true>(m, scr);
#pragma unroll
    for (int q = 0; q < QB; ++q) z[q] = m_run[q] == -INFINITY ? 0.f : z_run[q] * expf(m_run[q] - m[q]);
    block_reduce<QB, false>(z, scr);
    // dI(u) = c(u) p(u) sum(target) - T(u), in place of I
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      float lsum = 0.f;
      const float S = qst[q * 8 + kStS];
      const bool any = m[q] != -INFINITY;
      const float lz = any ? logf(z[q]) : 0.f;
      const float inv_z = any ? 1.f / z[q] : 0.f;
      for (int u = tid; u < n_u; u += kThreads) {
        const float c = mult(q, u);
        const float I = Iu[q * n_c + u];
        const float T = Tu[q * n_c + ulist[u]];
        float dI = 0.f;
        if (c > 0.f) {
          dI = c * expf(I - m[q]) * inv_z * S - T;
          if (T > 0.f) lsum += T * (I - m[q] - lz);
        }
        Iu[q * n_c + u] = dI;
      }
      lsum = warp_sum(lsum);
      if (lane == 0 && lsum != 0.f) atomicAdd(&qst[q * 8 + kStLoss], -lsum);
    }
  }
  __syncthreads();

  // ---- pass B: G from the signs, dQ^T += K^T G^T, dK^T = Q^T G ------------------------
  // G's weight per row: w, or 1 where |w| < 2^-60 (there the Q row is zeroed,
  // so that the row adds nothing to dK^T, and dq_I is scaled by w at the end)
  tmem_wait_st();                                     // the sign words are in TMEM
  if (tid < kRows) {
    const bool tiny = fabsf(wr[tid]) < kTinyW;
    wg[tid] = tiny ? 1.f : wr[tid];
    if (tiny) {
#pragma unroll
      for (int ch = 0; ch < 16; ++ch)
        *reinterpret_cast<uint4*>(sm + Layout::Q + sw_off(tid, ch)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // dK^T of tile it drained from TMEM (buffer it & 1): quad transposes give
  // lane 4a+b four consecutive d of slot 4k+b, so each vector reduction of a
  // warp covers 128 contiguous bytes of four block rows
  // Warp 0's thread 0 issues the products and is held until the tensor core
  // has taken them, so warp 0 drains nothing: the other three warps of its
  // lane quarter (column groups 1-3) share its eight 4-column blocks.
  auto drain_cols = [&](int it, int cgs, uint32_t blocks) {
    uint32_t v[32];
    tmem_ld32_wait(tmem + lane_base + (uint32_t)(it & 1) * 128 + cgs * 32, v);
    const int u0 = it * kSlots + cgs * 32;
    float* dk_q = dk_b + qd * 32 + 4 * (lane >> 2);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (!((blocks >> k) & 1u)) continue;
      float x[4] = {__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                    __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3])};
      quad_transpose4(x);
      const int u = u0 + 4 * k + (lane & 3);
      if (u < n_u) red_add_v4(dk_q + (long long)ulist[u] * kDI, x[0], x[1], x[2], x[3]);
    }
  };
  auto drain_dk = [&](int it) {
    if (warp == 0) return;
    drain_cols(it, cg, 0xFFu);
    if (qd == 0) drain_cols(it, 0, cg == 1 ? 0x07u : cg == 2 ? 0x38u : 0xC0u);
  };
  bool fail = false;                                 // a per-warp wait of this thread gave up
  if (ok && ntiles > 0) {
    stage(0, 0);
    if (ntiles > 1) stage(1, 1);
  }
  for (int it = 0; it < ntiles && ok; ++it) {
    // tile it-1's products are complete: G and KV buffer (it+1) & 1 are free
    if (it > 0) {
      const bool k_ok = __all_sync(0xffffffffu, mbar_wait(bar_dk, (it - 1) & 1));
      fail |= !k_ok;
      if (k_ok && it + 1 < ntiles) stage(it + 1, (it + 1) & 1);
    }
    if (!fail) {
      fence_after();
      const uint32_t signs = tmem_ld1_wait(tmem + lane_base + kColMask + it * 4 + cg);
      const int u = it * kSlots + r;
      const float dI = u < n_u ? Iu[myq * n_c + u] : 0.f;
      const float4* w4 = reinterpret_cast<const float4*>(wg + cg * 32);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const float4 wa = w4[2 * c8], wb = w4[2 * c8 + 1];
        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = (signs >> (c8 * 8 + e)) & 1u ? dI * wv[e] : 0.f;
        store_hi_lo8(GH, GL, sw_off(r, cg * 4 + c8), g);
      }
    }
    // tile it's rows (tile it+1's, staged above, may still be in flight)
    if (it + 1 < ntiles) cp_wait<1>();
    else cp_wait<0>();
    fence_proxy_async_smem();
    fence_before();
    ok = __syncthreads_and(!fail);
    if (!ok) { site = kSiteLossG; break; }
    if (tid == 0) {
      fence_after();
      const uint32_t ga = smem_addr(GH), la = smem_addr(GL);
      const uint32_t ka = smem_addr(sm + Layout::KV + (it & 1) * 2 * kBlk);
      const uint32_t qa = smem_addr(sm + Layout::Q);
      // dQ^T [d, rows] += K^T [d, slots] G^T [slots, rows]: A = K tile and B = G
      // read MN-major (16 slot lines per K step).  (G's lo part is needed here
      // too: a peaked student softmax leaves one slot with |G| near |w|, whose
      // bf16 rounding alone moved dq_I by 1e-2.)
      constexpr uint32_t idesc_q = idesc_bf16_f32_major(kDI, kRows, 1, 1);
#pragma unroll
      for (int k = 0; k < kSlots / 16; ++k) {
        const uint64_t a = sw128_desc_mn(ka + k * 2048, kBlk);
        mma_bf16_ss(tmem + kColDQ, a, sw128_desc_mn(ga + k * 2048, kBlk), idesc_q,
                    (it > 0 || k > 0) ? 1u : 0u);
        mma_bf16_ss(tmem + kColDQ, a, sw128_desc_mn(la + k * 2048, kBlk), idesc_q, 1u);
      }
      // dK^T [d, slots] = Q^T [d, rows] G [rows, slots] into buffer it & 1: A = Q
      // read MN-major, B = G read K-major (its slot lines hold the rows
      // contiguously); the TMEM lane is then d
      constexpr uint32_t idesc_k = idesc_bf16_f32_major(kDI, kSlots, 1, 0);
      const uint32_t col_k = (uint32_t)(it & 1) * 128;
#pragma unroll
      for (int k = 0; k < kRows / 16; ++k) {
        const uint32_t boff = (k >> 2) * kBlk + (k & 3) * 32;
        const uint64_t aq = sw128_desc_mn(qa + k * 2048, kBlk);
        mma_bf16_ss(tmem + col_k, aq, sw128_desc(ga + boff), idesc_k, k > 0 ? 1u : 0u);
        mma_bf16_ss(tmem + col_k, aq, sw128_desc(la + boff), idesc_k, 1u);
      }
      mma_commit(bar_dk);
    }
    // the previous tile's dK^T is added into dk_I while the tensor core forms
    // this tile's products
    if (it > 0) drain_dk(it - 1);
    fence_before();
  }
  if (ok && ntiles > 0) {
    // the last tile's products: then its dK^T, and dQ^T is complete
    const bool k_ok = __all_sync(0xffffffffu, mbar_wait(bar_dk, (ntiles - 1) & 1));
    if (k_ok) {
      fence_after();
      drain_dk(ntiles - 1);
    }
    ok = __syncthreads_and(k_ok);
    if (!ok) site = kSiteLossG;
  }
  cp_async_wait_all_();                               // no copy in flight past this point
  if (!ok && tid == 0) set_status(status, kDevTimeout, site);

  // ---- epilogue: dq_I rows and dw = q_I . dq_I / w, from dQ^T; loss ---------------------
  // thread (d = its TMEM lane, 32 rows): dQ^T[d][rows] and q_I[rows][d]
  uint32_t v[32];
  if (ok) {
    fence_after();
    if (ntiles > 0) {
      tmem_ld32_wait(tmem + lane_base + kColDQ + cg * 32, v);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = 0u;
    }
    const long long qrow0 = ((long long)bi * sq + t0) * H_I;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float p16[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int row = cg * 32 + h2 * 16 + c;
        const bool live = t0 + row / H_I < sq;
        const float qv = live ? __bfloat162float(q_I[(qrow0 + row) * kDI + r]) : 0.f;
        p16[c] = qv * __uint_as_float(v[h2 * 16 + c]);
      }
      const float s = lane_transpose_sum16(p16);
      if (lane < 16) red[qd * kRows + cg * 32 + h2 * 16 + lane] = s;
    }
  }
  __syncthreads();
  if (ok && tid < kRows) {
    const int q = tid / H_I, t = t0 + q;
    if (t < sq) {
      const float s = (red[tid] + red[kRows + tid]) + (red[2 * kRows + tid] + red[3 * kRows + tid]);
      dw[((long long)bi * sq + t) * H_I + tid % H_I] = s / wg[tid];
      if (tid % H_I == 0) loss[(long long)bi * sq + t] = qst[q * 8 + kStLoss];
    }
  }
  // dq_I rows: staged in G hi|lo (free: the last products have completed),
  // then one bulk copy of the block's contiguous rows instead of plain
  // stores queued behind the dk_I reductions
  if (ok) {
    float* stg = reinterpret_cast<float*>(GH);       // [128 rows][128 d] fp32 = 64 KB
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int row = cg * 32 + c;
      const float g = __uint_as_float(v[c]);
      stg[row * kDI + r] = wg[row] == wr[row] ? g : g * wr[row];
    }
    fence_proxy_async_smem();
  }
  fence_before();
  __syncthreads();
  if (ok && tid == 0) {
    const int nrows = min(QB, sq - t0) * H_I;
    bulk_store(dq_I + ((long long)bi * sq + t0) * H_I * kDI, GH, (uint32_t)nrows * kDI * 4u);
    bulk_commit();
    bulk_wait_read_all();      // the copy has read the staging before the CTA exits
  }
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace ilt

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_loss() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
size_t indexer_loss_tc_smem(int QB, int n_c) {
  const int NW = (QB + 3) / 4;
  return 1024 + ilt::Layout::DYN + (size_t)n_c * NW * 8 + (size_t)n_c * 4 +
         (size_t)2 * QB * n_c * 4;
}
}  // namespace

// bf16, d_I = 128 and H_I in {32, 64} (128 / H_I queries per CTA), with the
// union lists of n_c entries within shared memory.
bool indexer_loss_tc_supported(int H_I, int d_I, int n_c) {
  if (d_I != ilt::kDI || !(H_I == 32 || H_I == 64)) return false;
  if (encode_fn_loss() == nullptr) return false;
  if (n_c > 4096) return false;                 // 32 tiles of sign words in TMEM
  return indexer_loss_tc_smem(ilt::kRows / H_I, n_c) <= 227 * 1024;
}

cudaError_t launch_indexer_loss_tc(const void* q_I, const void* k_I, const float* w,
                                   const int32_t* idx, const float* target, float* loss,
                                   float* dq_I, float* dk_I, float* dw, int b, int sq, int H_I,
                                   int n_c, int ratio, int K, int* status, cudaStream_t s) {
  auto encode = encode_fn_loss();
  if (encode == nullptr) return cudaErrorNotSupported;
  cudaError_t e = launch_zero_f32(dk_I, (size_t)b * n_c * ilt::kDI, s);
  if (e != cudaSuccess) return e;
  CUtensorMap tq;
  const cuuint64_t dims[2] = {(cuuint64_t)ilt::kDI, (cuuint64_t)b * sq * H_I};
  const cuuint64_t strides[1] = {(cuuint64_t)ilt::kDI * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)ilt::kRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_I), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int QB = ilt::kRows / H_I;
  const size_t smem = indexer_loss_tc_smem(QB, n_c);
  const unsigned grid = (unsigned)(((sq + QB - 1) / QB) * b);   // heaviest blocks first
#define CSA_LOSS_TC(QQ)                                                                       \
  {                                                                                           \
    auto k = ilt::indexer_loss_tc_kernel<QQ>;                                                 \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);     \
    if (e != cudaSuccess) return e;                                                           \
    k<<<grid, ilt::kThreads, smem, s>>>(tq, (const __nv_bfloat16*)q_I,                        \
                                        (const __nv_bfloat16*)k_I, w, idx, target, loss,      \
                                        dq_I, dk_I, dw, sq, n_c, ratio, K, status);           \
    count_launches(1);                                                                        \
  }
  if (QB == 2) CSA_LOSS_TC(2)
  else CSA_LOSS_TC(4)
#undef CSA_LOSS_TC
  return cudaGetLastError();
}

}  // namespace csa
