// Indexer training path: the distillation teacher from the attention LSE,
// and the student's KL loss with its gradients through a rescoring of the
// selected entries.
//
// "Refactor Deepseek v4 to use Attention Gym's Compressed Sparse Attention"
// (indexer distillation): the teacher of query t over its selected entries
// is exp(logit - lse) summed over the heads and L1-normalized, lse being the
// attention's per-head LSE (window, selected entries and sink); the student
// is a second pass of the indexer over the selected entries only.  "Add
// unfused SBHD compressed sparse attention" (review of the teacher
// normalization): one common per-row shift keeps the mass from underflowing
// and cancels in the normalization; the KL gradient with respect to the
// student scores is predict * sum(target) - target.
//
// Both calls run one CTA per query.  bf16 rows with d (d_I) a multiple of 16
// go through warp-level MMAs (mma.sync m16n8k16, fp32 accumulate) over
// chunks of 64 selected slots gathered into shared memory; other shapes and
// fp32 inputs use a CUDA-core kernel with the same arithmetic in fp32.
//
// Teacher: per slot s, m_s = max_h a_hs and T'_s = sum_h 2^(a_hs - m_s) with
// a = logit*log2e - lse*log2e; at the end c = max_s m_s and
// target_s = T'_s 2^(m_s - c) / sum_s' T'_s' 2^(m_s' - c).
// Student: I_s = sum_h w_h max(0, D_hs) with D = q_I k_I[j_s]^T; then
// dI = softmax(I) * sum(target) - target, G_hs = dI_s w_h [D_hs > 0],
// dq_I = G K, dw_h = sum_s dI_s max(0, D_hs), dk_I[j_s] += (G^T Q_I)_s (fp32
// vector atomics; repeated blocks and every selecting query sum).  G enters
// the two products as bf16 hi + lo pairs (about 16 significant bits).
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "warp_mma.cuh"

namespace csa {
namespace {

constexpr int kTrChunk = 64;     // selected slots per shared-memory chunk
constexpr int kTrThreads = 128;  // 4 warps; warp w owns slots 16w..16w+15 of a chunk

// First slot of the ci-th chunk a CTA visits.  Index rows are sorted, so
// neighbouring queries select mostly the same blocks in the same order; CTAs
// start at different chunks (rotated by the query index) so that the ones
// running together do not all read the same few rows, which would pile the
// requests onto one L2 slice.
__device__ __forceinline__ int chunk_start(int ci, int K) {
  const int n = (K + kTrChunk - 1) / kTrChunk;
  return ((ci + (int)blockIdx.x) % n) * kTrChunk;
}

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kTrThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// Gather rows `rows[c0 + r]` of a [*, D] bf16 matrix into a [64][LD] shared
// tile with 16-byte copies; invalid slots get zero rows (their results are
// dropped, and zeros keep the products finite).
template <int D, int LD>
__device__ __forceinline__ void gather_rows(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                            const int* rows, int c0, int K) {
  for (int e = threadIdx.x; e < kTrChunk * (D / 8); e += kTrThreads) {
    const int r = e / (D / 8), c8 = e % (D / 8);
    const int s = c0 + r;
    if (s < K && rows[s] >= 0)
      cp_async16(dst + r * LD + c8 * 8, src + (long long)rows[s] * D + c8 * 8);
    else
      *reinterpret_cast<uint4*>(dst + r * LD + c8 * 8) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  cp_async_wait_all();
}

// acc[mt][nt] = A[mt*16.., :] x B[16w + nt*8.., :]^T over K = D: A rows of
// `As` ([MT*16][LD]), B rows of `Bs` ([64][LD]) for this warp's 16 slots.
template <int D, int LD, int MT>
__device__ __forceinline__ void rows_x_slots(float (&acc)[MT][2][4], const __nv_bfloat16* As,
                                             const __nv_bfloat16* Bs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t b[4];
    ldsm_x4(b, Bs + (warp * 16 + (lane & 7) + ((lane >> 4) << 3)) * LD + kk * 16 +
                   ((lane >> 3) & 1) * 8);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t a[4];
      ldsm_x4(a, As + (mt * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
      mma_bf16(acc[mt][0], a, b[0], b[1]);
      mma_bf16(acc[mt][1], a, b[2], b[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// teacher
// ---------------------------------------------------------------------------

template <int D, int HP>
__global__ void __launch_bounds__(kTrThreads) teacher_mma_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
    const int32_t* __restrict__ idx, const float* __restrict__ lse, float scale,
    float* __restrict__ target, int sq, int H, int n_c, int ratio, int K) {
  constexpr int LD = D + 8, MT = HP / 16;
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem);   // [HP][LD]
  __nv_bfloat16* Ks = Qs + HP * LD;                              // [64][LD]
  float* lse2 = reinterpret_cast<float*>(Ks + kTrChunk * LD);    // [HP]
  float* red = lse2 + HP;                                        // [32]
  float* mS = red + 32;                                          // [K]
  float* TS = mS + K;                                            // [K]
  int* rows = reinterpret_cast<int*>(TS + K);                    // [K]
  const int t = blockIdx.x, bi = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int vis = min((t + 1) / ratio, n_c);
  const long long row_q = (long long)bi * sq + t;
  const __nv_bfloat16* qt = q + row_q * H * D;
  for (int e = tid; e < HP * (D / 8); e += kTrThreads) {
    const int h = e / (D / 8), c8 = e % (D / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h < H) v = *reinterpret_cast<const uint4*>(qt + h * D + c8 * 8);
    *reinterpret_cast<uint4*>(Qs + h * LD + c8 * 8) = v;
  }
  for (int h = tid; h < HP; h += kTrThreads) lse2[h] = h < H ? lse[row_q * H + h] * kLog2e : INFINITY;
  const int32_t* ir = idx + row_q * K;
  for (int s = tid; s < K; s += kTrThreads) {
    const int j = ir[s];
    rows[s] = (j >= 0 && j < vis) ? sq + j : -1;
  }
  __syncthreads();
  const float sc2 = scale * kLog2e;
  const __nv_bfloat16* kv_b = kv + (long long)bi * (sq + n_c) * D;
  for (int ci = 0; ci * kTrChunk < K; ++ci) {
    const int c0 = chunk_start(ci, K);
    // a chunk without valid slots (the -1 tail of a short row) is skipped
    if (!__syncthreads_or(tid < kTrChunk && c0 + tid < K && rows[c0 + tid] >= 0)) continue;
    gather_rows<D, LD>(Ks, kv_b, rows, c0, K);
    __syncthreads();
    float acc[MT][2][4];
    rows_x_slots<D, LD, MT>(acc, Qs, Ks);
    // per slot (column): max and shifted sum over the heads (rows); padded
    // heads have lse2 = +inf, so they contribute 2^-inf = 0
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float m = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          m = fmaxf(m, fmaf(acc[mt][nt][cc], sc2, -lse2[mt * 16 + g]));
          m = fmaxf(m, fmaf(acc[mt][nt][cc + 2], sc2, -lse2[mt * 16 + g + 8]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          sum += exp2f(fmaf(acc[mt][nt][cc], sc2, -lse2[mt * 16 + g]) - m);
          sum += exp2f(fmaf(acc[mt][nt][cc + 2], sc2, -lse2[mt * 16 + g + 8]) - m);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const int s = c0 + warp * 16 + nt * 8 + 2 * c + cc;
        if (g == 0 && s < K) {
          mS[s] = m;
          TS[s] = sum;
        }
      }
    __syncthreads();
  }
  // one shift for the row, then the L1 normalization
  float mx = -INFINITY;
  for (int s = tid; s < K; s += kTrThreads)
    if (rows[s] >= 0) mx = fmaxf(mx, mS[s]);
  mx = block_reduce(mx, red, true);
  float tot = 0.f;
  for (int s = tid; s < K; s += kTrThreads) {
    const float v = rows[s] >= 0 ? TS[s] * exp2f(mS[s] - mx) : 0.f;
    TS[s] = v;
    tot += v;
  }
  tot = block_reduce(tot, red, false);
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  float* out = target + row_q * K;
  for (int s = tid; s < K; s += kTrThreads) out[s] = TS[s] * inv;
}

template <typename T>
__global__ void __launch_bounds__(kTrThreads) teacher_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ kv, const int32_t* __restrict__ idx,
    const float* __restrict__ lse, float scale, float* __restrict__ target, int sq, int H, int d,
    int n_c, int ratio, int K) {
  extern __shared__ __align__(16) float fsm[];
  float* red = fsm;              // [32]
  float* mS = red + 32;          // [K]
  float* TS = mS + K;            // [K]
  int* rows = reinterpret_cast<int*>(TS + K);
  const int t = blockIdx.x, bi = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vis = min((t + 1) / ratio, n_c);
  const long long row_q = (long long)bi * sq + t;
  const int32_t* ir = idx + row_q * K;
  for (int s = tid; s < K; s += kTrThreads) {
    const int j = ir[s];
    rows[s] = (j >= 0 && j < vis) ? sq + j : -1;
  }
  __syncthreads();
  const T* qt = q + row_q * H * d;
  const T* kv_b = kv + (long long)bi * (sq + n_c) * d;
  const float sc2 = scale * kLog2e;
  // one warp per slot; heads one after the other
  for (int s = warp; s < K; s += kTrThreads / 32) {
    if (rows[s] < 0) continue;
    const T* kr = kv_b + (long long)rows[s] * d;
    float m = -INFINITY, sum = 0.f;
    for (int h = 0; h < H; ++h) {
      float dot = 0.f;
      for (int e = lane; e < d; e += 32) dot = fmaf(to_f(qt[h * d + e]), to_f(kr[e]), dot);
      dot = warp_sum(dot);
      const float a = fmaf(dot, sc2, -lse[row_q * H + h] * kLog2e);
      const float mn = fmaxf(m, a);
      sum = sum * exp2f(m - mn) + exp2f(a - mn);
      m = mn;
    }
    if (lane == 0) {
      mS[s] = m;
      TS[s] = sum;
    }
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int s = tid; s < K; s += kTrThreads)
    if (rows[s] >= 0) mx = fmaxf(mx, mS[s]);
  mx = block_reduce(mx, red, true);
  float tot = 0.f;
  for (int s = tid; s < K; s += kTrThreads) {
    const float v = rows[s] >= 0 ? TS[s] * exp2f(mS[s] - mx) : 0.f;
    TS[s] = v;
    tot += v;
  }
  tot = block_reduce(tot, red, false);
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  for (int s = tid; s < K; s += kTrThreads) target[row_q * K + s] = TS[s] * inv;
}

// ---------------------------------------------------------------------------
// student KL loss and gradients
// ---------------------------------------------------------------------------

// Row softmax over the valid slots of Is, the KL loss against `tg`, and
// dI = p * sum(target) - target into dIs (0 at invalid slots).  Returns the
// loss (valid in every thread).
__device__ __forceinline__ float kl_row(const float* Is, const int* blk, const float* tg, float* dIs,
                                        int K, float* red) {
  const int tid = threadIdx.x;
  float mx = -INFINITY;
  for (int s = tid; s < K; s += kTrThreads)
    if (blk[s] >= 0) mx = fmaxf(mx, Is[s]);
  mx = block_reduce(mx, red, true);
  float se = 0.f, ts = 0.f;
  for (int s = tid; s < K; s += kTrThreads)
    if (blk[s] >= 0) {
      se += __expf(Is[s] - mx);
      ts += tg[s];
    }
  se = block_reduce(se, red, false);
  ts = block_reduce(ts, red, false);
  const float lse = mx + logf(se);
  float loss = 0.f;
  for (int s = tid; s < K; s += kTrThreads) {
    float di = 0.f;
    if (blk[s] >= 0) {
      const float logp = Is[s] - lse;
      const float tv = tg[s];
      if (tv > 0.f) loss += tv * (logf(tv) - logp);
      di = __expf(logp) * ts - tv;
    }
    dIs[s] = di;
  }
  return block_reduce(loss, red, false);
}

// Three CTAs per SM (168 registers, a few spilled) beat two at 179 registers:
// the kernel is bound by the latency of its warp-level MMAs and gathers.
template <int DI, int HIP>
__global__ void __launch_bounds__(kTrThreads, 3) student_mma_kernel(
    const __nv_bfloat16* __restrict__ q_I, const __nv_bfloat16* __restrict__ k_I,
    const float* __restrict__ w, const int32_t* __restrict__ idx, const float* __restrict__ target,
    float* __restrict__ loss, float* __restrict__ dq_I, float* __restrict__ dk_I,
    float* __restrict__ dw, int sq, int H_I, int n_c, int ratio, int K) {
  constexpr int LD = DI + 8, MT = HIP / 16, LG = kTrChunk + 8;
  constexpr int NQ = DI / 32;          // dq n8-tiles per warp (warps split d_I)
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem);   // [HIP][LD]
  __nv_bfloat16* Ks = Qs + HIP * LD;                             // [64][LD]
  __nv_bfloat16* Gh = Ks + kTrChunk * LD;                        // [HIP][LG]
  __nv_bfloat16* Gl = Gh + HIP * LG;                             // [HIP][LG]
  float* ws = reinterpret_cast<float*>(Gl + HIP * LG);           // [HIP]
  float* red = ws + HIP;                                         // [32]
  float* dwp = red + 32;                                         // [4][HIP]
  float* Is = dwp + 4 * HIP;                                     // [K]
  float* dIs = Is + K;                                           // [K]
  float* tg = dIs + K;                                           // [K]
  int* blk = reinterpret_cast<int*>(tg + K);                     // [K]
  const int t = blockIdx.x, bi = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int vis = min((t + 1) / ratio, n_c);
  const long long row_q = (long long)bi * sq + t;
  const __nv_bfloat16* qt = q_I + row_q * H_I * DI;
  for (int e = tid; e < HIP * (DI / 8); e += kTrThreads) {
    const int h = e / (DI / 8), c8 = e % (DI / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h < H_I) v = *reinterpret_cast<const uint4*>(qt + h * DI + c8 * 8);
    *reinterpret_cast<uint4*>(Qs + h * LD + c8 * 8) = v;
  }
  for (int h = tid; h < HIP; h += kTrThreads) ws[h] = h < H_I ? w[row_q * H_I + h] : 0.f;
  const int32_t* ir = idx + row_q * K;
  for (int s = tid; s < K; s += kTrThreads) {
    const int j = ir[s];
    blk[s] = (j >= 0 && j < vis) ? j : -1;
    tg[s] = target[row_q * K + s];
  }
  __syncthreads();
  const __nv_bfloat16* k_b = k_I + (long long)bi * n_c * DI;

  // ---- pass A: student scores of the selected slots ------------------------
  for (int ci = 0; ci * kTrChunk < K; ++ci) {
    const int c0 = chunk_start(ci, K);
    if (!__syncthreads_or(tid < kTrChunk && c0 + tid < K && blk[c0 + tid] >= 0)) continue;
    gather_rows<DI, LD>(Ks, k_b, blk, c0, K);
    __syncthreads();
    float acc[MT][2][4];
    rows_x_slots<DI, LD, MT>(acc, Qs, Ks);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float v = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          v = fmaf(ws[mt * 16 + g], fmaxf(acc[mt][nt][cc], 0.f), v);
          v = fmaf(ws[mt * 16 + g + 8], fmaxf(acc[mt][nt][cc + 2], 0.f), v);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int s = c0 + warp * 16 + nt * 8 + 2 * c + cc;
        if (g == 0 && s < K) Is[s] = v;
      }
    __syncthreads();
  }

  // ---- KL loss and dI ----------------------------------------------------------
  const float lrow = kl_row(Is, blk, tg, dIs, K, red);
  if (tid == 0) loss[row_q] = lrow;
  __syncthreads();

  // ---- pass B: gradients -------------------------------------------------------
  float dqa[MT][NQ][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NQ; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) dqa[mt][nt][e] = 0.f;
  float dwl[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) dwl[mt][0] = dwl[mt][1] = 0.f;
  float* dk_b = dk_I + (long long)bi * n_c * DI;
  for (int ci = 0; ci * kTrChunk < K; ++ci) {
    const int c0 = chunk_start(ci, K);
    if (!__syncthreads_or(tid < kTrChunk && c0 + tid < K && blk[c0 + tid] >= 0)) continue;
    gather_rows<DI, LD>(Ks, k_b, blk, c0, K);
    __syncthreads();
    {
      float acc[MT][2][4];
      rows_x_slots<DI, LD, MT>(acc, Qs, Ks);
      // G = dI * w * [D > 0] as bf16 hi + lo; dw partial sums
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int sl = warp * 16 + nt * 8 + 2 * c;       // chunk-local slot of element cc = 0
        const float d0 = c0 + sl < K ? dIs[c0 + sl] : 0.f;
        const float d1 = c0 + sl + 1 < K ? dIs[c0 + sl + 1] : 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int h = mt * 16 + g + hh * 8;
            const float x0 = acc[mt][nt][2 * hh], x1 = acc[mt][nt][2 * hh + 1];
            dwl[mt][hh] = fmaf(d0, fmaxf(x0, 0.f), fmaf(d1, fmaxf(x1, 0.f), dwl[mt][hh]));
            const float g0 = x0 > 0.f ? d0 * ws[h] : 0.f;
            const float g1 = x1 > 0.f ? d1 * ws[h] : 0.f;
            const __nv_bfloat162 hi = __floats2bfloat162_rn(g0, g1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(g0 - hf.x, g1 - hf.y);
            *reinterpret_cast<__nv_bfloat162*>(Gh + h * LG + sl) = hi;
            *reinterpret_cast<__nv_bfloat162*>(Gl + h * LG + sl) = lo;
          }
      }
    }
    __syncthreads();
    // dq_I += G K_chunk: rows = heads, k = slots, n = d_I (warp w: columns w*DI/4 ...)
#pragma unroll
    for (int ks = 0; ks < kTrChunk / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < NQ / 2; ++np) {
        uint32_t b[4];
        ldsm_x4_t(b, Ks + (ks * 16 + (lane & 15)) * LD + warp * (DI / 4) + np * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t ah[4], al[4];
          ldsm_x4(ah, Gh + (mt * 16 + (lane & 15)) * LG + ks * 16 + (lane >> 4) * 8);
          ldsm_x4(al, Gl + (mt * 16 + (lane & 15)) * LG + ks * 16 + (lane >> 4) * 8);
          mma_bf16(dqa[mt][2 * np], ah, b[0], b[1]);
          mma_bf16(dqa[mt][2 * np], al, b[0], b[1]);
          mma_bf16(dqa[mt][2 * np + 1], ah, b[2], b[3]);
          mma_bf16(dqa[mt][2 * np + 1], al, b[2], b[3]);
        }
      }
    }
    // dk_I rows of this warp's 16 slots: (G^T Q_I), k = heads, n = d_I
    {
      float acc2[DI / 8][4];
#pragma unroll
      for (int nt = 0; nt < DI / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc2[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < MT; ++ks) {
        uint32_t ah[4], al[4];
        const int ar = ks * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ac = warp * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(ah, Gh + ar * LG + ac);
        ldsm_x4_t(al, Gl + ar * LG + ac);
#pragma unroll
        for (int np = 0; np < DI / 16; ++np) {
          uint32_t b[4];
          ldsm_x4_t(b, Qs + (ks * 16 + (lane & 15)) * LD + np * 16 + (lane >> 4) * 8);
          mma_bf16(acc2[2 * np], ah, b[0], b[1]);
          mma_bf16(acc2[2 * np], al, b[0], b[1]);
          mma_bf16(acc2[2 * np + 1], ah, b[2], b[3]);
          mma_bf16(acc2[2 * np + 1], al, b[2], b[3]);
        }
      }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int s = c0 + warp * 16 + g + hh * 8;
        if (s < K && blk[s] >= 0) {
          float* dst = dk_b + (long long)blk[s] * DI + 2 * c;
#pragma unroll
          for (int nt = 0; nt < DI / 8; ++nt)
            red_add_v2(dst + nt * 8, acc2[nt][2 * hh], acc2[nt][2 * hh + 1]);
        }
      }
    }
    __syncthreads();
  }
  // dq_I rows (heads < H_I)
  float* dqt = dq_I + row_q * H_I * DI;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = mt * 16 + g + hh * 8;
      if (h < H_I) {
#pragma unroll
        for (int nt = 0; nt < NQ; ++nt)
          *reinterpret_cast<float2*>(dqt + h * DI + warp * (DI / 4) + nt * 8 + 2 * c) =
              make_float2(dqa[mt][nt][2 * hh], dqa[mt][nt][2 * hh + 1]);
      }
    }
  // dw: the 4 lanes of a row share g; then the 4 warps (disjoint slots)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float v = dwl[mt][hh];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (c == 0) dwp[warp * HIP + mt * 16 + g + hh * 8] = v;
    }
  __syncthreads();
  for (int h = tid; h < H_I; h += kTrThreads)
    dw[row_q * H_I + h] = (dwp[h] + dwp[HIP + h]) + (dwp[2 * HIP + h] + dwp[3 * HIP + h]);
}

template <typename T>
__global__ void __launch_bounds__(kTrThreads) student_simt_kernel(
    const T* __restrict__ q_I, const T* __restrict__ k_I, const float* __restrict__ w,
    const int32_t* __restrict__ idx, const float* __restrict__ target, float* __restrict__ loss,
    float* __restrict__ dq_I, float* __restrict__ dk_I, float* __restrict__ dw, int sq, int H_I,
    int d_I, int n_c, int ratio, int K) {
  extern __shared__ __align__(16) float fsm[];
  float* red = fsm;                  // [32]
  float* dqs = red + 32;             // [H_I][d_I]
  float* dws = dqs + H_I * d_I;      // [H_I]
  float* Is = dws + H_I;             // [K]
  float* dIs = Is + K;               // [K]
  float* tg = dIs + K;               // [K]
  int* blk = reinterpret_cast<int*>(tg + K);
  const int t = blockIdx.x, bi = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vis = min((t + 1) / ratio, n_c);
  const long long row_q = (long long)bi * sq + t;
  const int32_t* ir = idx + row_q * K;
  for (int s = tid; s < K; s += kTrThreads) {
    const int j = ir[s];
    blk[s] = (j >= 0 && j < vis) ? j : -1;
    tg[s] = target[row_q * K + s];
    Is[s] = 0.f;
  }
  for (int e = tid; e < H_I * d_I + H_I; e += kTrThreads) dqs[e] = 0.f;
  __syncthreads();
  const T* qt = q_I + row_q * H_I * d_I;
  const T* k_b = k_I + (long long)bi * n_c * d_I;
  const float* wt = w + row_q * H_I;
  for (int s = warp; s < K; s += kTrThreads / 32) {
    if (blk[s] < 0) continue;
    const T* kr = k_b + (long long)blk[s] * d_I;
    float v = 0.f;
    for (int h = 0; h < H_I; ++h) {
      float dot = 0.f;
      for (int e = lane; e < d_I; e += 32) dot = fmaf(to_f(qt[h * d_I + e]), to_f(kr[e]), dot);
      v = fmaf(wt[h], fmaxf(warp_sum(dot), 0.f), v);
    }
    if (lane == 0) Is[s] = v;
  }
  __syncthreads();
  const float lrow = kl_row(Is, blk, tg, dIs, K, red);
  if (tid == 0) loss[row_q] = lrow;
  __syncthreads();
  float* dk_b = dk_I + (long long)bi * n_c * d_I;
  for (int s = warp; s < K; s += kTrThreads / 32) {
    if (blk[s] < 0) continue;
    const T* kr = k_b + (long long)blk[s] * d_I;
    const float di = dIs[s];
    for (int h = 0; h < H_I; ++h) {
      float dot = 0.f;
      for (int e = lane; e < d_I; e += 32) dot = fmaf(to_f(qt[h * d_I + e]), to_f(kr[e]), dot);
      dot = warp_sum(dot);
      if (lane == 0) atomicAdd(&dws[h], di * fmaxf(dot, 0.f));
      if (dot > 0.f) {
        const float gg = di * wt[h];
        for (int e = lane; e < d_I; e += 32) {
          atomicAdd(&dqs[h * d_I + e], gg * to_f(kr[e]));
          atomicAdd(&dk_b[(long long)blk[s] * d_I + e], gg * to_f(qt[h * d_I + e]));
        }
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < H_I * d_I; e += kTrThreads) dq_I[row_q * H_I * d_I + e] = dqs[e];
  for (int h = tid; h < H_I; h += kTrThreads) dw[row_q * H_I + h] = dws[h];
}

int pad16(int x) { return (x + 15) / 16 * 16; }

}  // namespace

size_t indexer_teacher_smem(bool mma, int H, int d, int K) {
  if (mma) {
    const int HP = pad16(H) == 48 ? 64 : pad16(H);
    return (size_t)(HP + kTrChunk) * (d + 8) * 2 + (size_t)(HP + 32) * 4 + (size_t)K * 12;
  }
  return 32 * 4 + (size_t)K * 12;
}

size_t indexer_loss_smem(bool mma, int H_I, int d_I, int K) {
  if (mma) {
    const int HP = pad16(H_I) == 48 ? 64 : pad16(H_I);
    return (size_t)(HP + kTrChunk) * (d_I + 8) * 2 + (size_t)2 * HP * (kTrChunk + 8) * 2 +
           (size_t)(HP + 32 + 4 * HP) * 4 + (size_t)K * 16;
  }
  return (size_t)(32 + H_I * d_I + H_I) * 4 + (size_t)K * 16;
}

bool indexer_teacher_mma_ok(int H, int d) {
  return H <= 64 && (d == 64 || d == 128 || d == 256 || d == 512);
}
bool indexer_loss_mma_ok(int H_I, int d_I) { return H_I <= 64 && (d_I == 64 || d_I == 128); }

cudaError_t launch_indexer_teacher(const void* q, const void* kv, const int32_t* idx,
                                   const float* lse, float scale, float* target, int b, int sq,
                                   int H, int d, int n_c, int ratio, int K, bool bf16,
                                   cudaStream_t s) {
  dim3 grid((unsigned)sq, (unsigned)b);
  if (bf16 && indexer_teacher_mma_ok(H, d)) {
    const size_t smem = indexer_teacher_smem(true, H, d, K);
    const int HP = pad16(H) == 48 ? 64 : pad16(H);
#define CSA_TEACH(DD, PP)                                                                      \
  {                                                                                            \
    auto k = teacher_mma_kernel<DD, PP>;                                                       \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                         (int)smem);                                           \
    if (e != cudaSuccess) return e;                                                            \
    k<<<grid, kTrThreads, smem, s>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx,  \
                                     lse, scale, target, sq, H, n_c, ratio, K);                \
    count_launches(1);                                                                         \
    return cudaGetLastError();                                                                 \
  }
#define CSA_TEACH_D(DD) \
  if (HP == 16) CSA_TEACH(DD, 16) else if (HP == 32) CSA_TEACH(DD, 32) else CSA_TEACH(DD, 64)
    if (d == 64) CSA_TEACH_D(64)
    else if (d == 128) CSA_TEACH_D(128)
    else if (d == 256) CSA_TEACH_D(256)
    else CSA_TEACH_D(512)
#undef CSA_TEACH_D
#undef CSA_TEACH
  }
  const size_t smem = indexer_teacher_smem(false, H, d, K);
  if (bf16) {
    auto k = teacher_simt_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kTrThreads, smem, s>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx, lse,
                                     scale, target, sq, H, d, n_c, ratio, K);
  } else {
    auto k = teacher_simt_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kTrThreads, smem, s>>>((const float*)q, (const float*)kv, idx, lse, scale, target,
                                     sq, H, d, n_c, ratio, K);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_indexer_loss(const void* q_I, const void* k_I, const float* w,
                                const int32_t* idx, const float* target, float* loss, float* dq_I,
                                float* dk_I, float* dw, int b, int sq, int H_I, int d_I, int n_c,
                                int ratio, int K, bool bf16, cudaStream_t s) {
  cudaError_t e = launch_zero_f32(dk_I, (size_t)b * n_c * d_I, s);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)sq, (unsigned)b);
  if (bf16 && indexer_loss_mma_ok(H_I, d_I)) {
    const size_t smem = indexer_loss_smem(true, H_I, d_I, K);
    const int HP = pad16(H_I) == 48 ? 64 : pad16(H_I);
#define CSA_STUD(DD, PP)                                                                       \
  {                                                                                            \
    auto k = student_mma_kernel<DD, PP>;                                                       \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);      \
    if (e != cudaSuccess) return e;                                                            \
    k<<<grid, kTrThreads, smem, s>>>((const __nv_bfloat16*)q_I, (const __nv_bfloat16*)k_I, w, \
                                     idx, target, loss, dq_I, dk_I, dw, sq, H_I, n_c, ratio,  \
                                     K);                                                       \
    count_launches(1);                                                                         \
    return cudaGetLastError();                                                                 \
  }
#define CSA_STUD_D(DD) \
  if (HP == 16) CSA_STUD(DD, 16) else if (HP == 32) CSA_STUD(DD, 32) else CSA_STUD(DD, 64)
    if (d_I == 64) CSA_STUD_D(64)
    else CSA_STUD_D(128)
#undef CSA_STUD_D
#undef CSA_STUD
  }
  const size_t smem = indexer_loss_smem(false, H_I, d_I, K);
  if (bf16) {
    auto k = student_simt_kernel<__nv_bfloat16>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kTrThreads, smem, s>>>((const __nv_bfloat16*)q_I, (const __nv_bfloat16*)k_I, w, idx,
                                     target, loss, dq_I, dk_I, dw, sq, H_I, d_I, n_c, ratio, K);
  } else {
    auto k = student_simt_kernel<float>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kTrThreads, smem, s>>>((const float*)q_I, (const float*)k_I, w, idx, target, loss,
                                     dq_I, dk_I, dw, sq, H_I, d_I, n_c, ratio, K);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
