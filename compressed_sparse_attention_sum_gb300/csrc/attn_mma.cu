// Sparse MQA forward/backward for bf16 on the warp-level tensor-core path
// (mma.sync m16n8k16, fp32 accumulate).
//
// One CTA per (query row, group of up to 16*MT heads).  The query's slot rows
// (window rows, then the valid selected compressed rows of the compact KV
// buffer) are gathered tile by tile into shared memory with 16-byte cp.async
// copies; the same KV tile serves as K (scores) and as V (values), since K
// and V are one shared row ("Add unfused SBHD compressed sparse attention",
// unfused sparse core: one kv_full gathered once, both einsums on it).
//
// Forward per tile: S = Q K^T (warps split slots), online softmax with the
// sink as the initial running state (m = sink, l = 1) so it enters only the
// denominator, P -> bf16 in shared memory, O += P V (warps split d).
// Backward: a first pass over the slot tiles forms D = sum_i p_i dP_i (equal
// to dO.O, but without the bf16 rounding of the stored O); the second pass
// recomputes S and dP = dO V^T from one KV fragment, P = exp(S - lse) (the
// forward LSE includes the sink), dS = P (dP - D), dQ += dS K in registers,
// and dKV_tile = P^T dO + dS^T Q, which sums over the heads inside the MMA
// before one fp32 vector atomic per element of the compact [b*n_kv, d]
// buffer ("Add the min-memory DSA attention kernels": scatter of selected
// gradients with repeated indices accumulates in fp32).  P and dS enter
// these products as bf16 hi + lo pairs (x = hi + lo, hi = bf16(x),
// lo = bf16(x - hi)), about 16 significant bits, so the sums over thousands
// of queries stay within the fp32-accumulation error of the method.
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "warp_mma.cuh"

namespace csa {

// Gather slot rows [base, base+NS) of the query into a padded smem tile.
template <int D, int NS, int LD, int NT>
__device__ __forceinline__ void gather_tile(__nv_bfloat16* dst, const __nv_bfloat16* kv_b,
                                            const int* rows, int base, int count) {
  constexpr int CH = D / 8;
  for (int ci = threadIdx.x; ci < NS * CH; ci += NT) {
    const int r = ci / CH, cc = ci % CH;
    const int p = base + r;
    const int row = rows[p < count ? p : 0];
    cp_async16(dst + r * LD + cc * 8, kv_b + (long long)row * D + cc * 8);
  }
}

// Load ROWS x D bf16 rows (heads h0.. of one query) into padded smem; rows
// past H are zero.
template <int D, int ROWS, int LD, int NT>
__device__ __forceinline__ void load_heads(__nv_bfloat16* dst, const __nv_bfloat16* src, int h0,
                                           int H) {
  constexpr int CH = D / 8;
  for (int ci = threadIdx.x; ci < ROWS * CH; ci += NT) {
    const int r = ci / CH, cc = ci % CH;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h0 + r < H) v = *reinterpret_cast<const uint4*>(src + (long long)(h0 + r) * D + cc * 8);
    *reinterpret_cast<uint4*>(dst + r * LD + cc * 8) = v;
  }
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------
template <int D, int MT>
struct FwdCfg {
  static constexpr int NW = 4 * MT;
  static constexpr int NT = NW * 32;
  static constexpr int NS = D <= 128 ? 64 : 32;
  static constexpr int ROWS = 16 * MT;
  static constexpr int LDQ = D + 8;
  static constexpr int LDS = NS + 4;
  static constexpr int LDP = NS + 8;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + ROWS * LDQ * 2;
  static constexpr int OFF_S = OFF_KV + 2 * NS * LDQ * 2;
  static constexpr int OFF_P = OFF_S + ROWS * LDS * 4;
  static constexpr int OFF_STAT = OFF_P + ROWS * LDP * 2;
  static constexpr int OFF_ROWS = OFF_STAT + 3 * ROWS * 4;
};

template <int D, int MT>
__global__ void __launch_bounds__(FwdCfg<D, MT>::NT) attn_fwd_mma(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
    const int32_t* __restrict__ idx, const float* __restrict__ sink, float scale,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int sq, int H, int n_c, int ratio,
    int window, int K, const int32_t* __restrict__ doc, int tb) {
  using C = FwdCfg<D, MT>;
  constexpr int NS = C::NS, LDQ = C::LDQ, LDS = C::LDS, LDP = C::LDP, NT = C::NT, NW = C::NW;
  constexpr int NQ = NS / 32;      // n8-tiles per warp in the score phase
  constexpr int NO = D / 32;       // n8-tiles per warp in the PV phase
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_Q);
  __nv_bfloat16* KVs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_KV);
  float* Ss = reinterpret_cast<float*>(smem + C::OFF_S);
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_P);
  float* m_s = reinterpret_cast<float*>(smem + C::OFF_STAT);
  float* l_s = m_s + C::ROWS;
  float* a_s = l_s + C::ROWS;
  int* rows = reinterpret_cast<int*>(smem + C::OFF_ROWS);
  __shared__ int s_count;

  const int t = tb + (int)blockIdx.x, bi = blockIdx.y, h0 = blockIdx.z * C::ROWS;
  const int tid = threadIdx.x, w = tid / 32, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  const int n_kv = sq + n_c;
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * D;

  if (w == 0) {
    const int c = build_slots_warp(rows, idx ? idx + ((long long)bi * sq + t) * K : nullptr, K, t,
                                   sq, n_c, ratio, window, doc ? doc + (long long)bi * sq : nullptr);
    if (lane == 0) s_count = c;
  }
  load_heads<D, C::ROWS, LDQ, NT>(Qs, q + ((long long)bi * sq + t) * H * D, h0, H);
  for (int r = tid; r < C::ROWS; r += NT) {
    const int h = h0 + r;
    const bool hs = sink != nullptr && h < H;
    m_s[r] = hs ? sink[h] * kLog2e : -INFINITY;
    l_s[r] = hs ? 1.f : 0.f;
  }
  __syncthreads();
  const int count = s_count;
  const int ntiles = (count + NS - 1) / NS;
  const float sc2 = scale * kLog2e;

  gather_tile<D, NS, LDQ, NT>(KVs, kv_b, rows, 0, count);
  cp_async_commit();

  float oacc[NO][4];
#pragma unroll
  for (int n = 0; n < NO; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;

  const int mt_s = w % MT, grp = w / MT;    // score phase: 16 heads x NS/4 slots
  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait_all();
    __syncthreads();
    if (it + 1 < ntiles) {
      gather_tile<D, NS, LDQ, NT>(KVs + ((it + 1) & 1) * NS * LDQ, kv_b, rows, (it + 1) * NS,
                                  count);
      cp_async_commit();
    }
    const __nv_bfloat16* KT = KVs + (it & 1) * NS * LDQ;
    // ---- S = Q K^T -------------------------------------------------------
    {
      float sacc[NQ][4];
#pragma unroll
      for (int n = 0; n < NQ; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
      const int n0 = grp * (NS / 4);
#pragma unroll 4
      for (int k = 0; k < D / 16; ++k) {
        uint32_t a[4];
        ldsm_x4(a, Qs + (mt_s * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDQ + k * 16 +
                       8 * (lane >> 4));
        if constexpr (NQ == 2) {
          uint32_t bb[4];
          ldsm_x4(bb, KT + (n0 + (lane & 7) + 8 * (lane >> 4)) * LDQ + k * 16 +
                          8 * ((lane >> 3) & 1));
          mma_bf16(sacc[0], a, bb[0], bb[1]);
          mma_bf16(sacc[1], a, bb[2], bb[3]);
        } else {
          uint32_t bb[2];
          ldsm_x2(bb, KT + (n0 + (lane & 7)) * LDQ + k * 16 + 8 * ((lane >> 3) & 1));
          mma_bf16(sacc[0], a, bb[0], bb[1]);
        }
      }
#pragma unroll
      for (int n = 0; n < NQ; ++n) {
        const int col = n0 + n * 8 + 2 * cq;
        float* r0 = Ss + (mt_s * 16 + g) * LDS + col;
        float* r1 = r0 + 8 * LDS;
        r0[0] = sacc[n][0] * sc2;
        r0[1] = sacc[n][1] * sc2;
        r1[0] = sacc[n][2] * sc2;
        r1[1] = sacc[n][3] * sc2;
      }
    }
    __syncthreads();
    // ---- online softmax (log2 domain) -------------------------------------
    {
      const int base = it * NS;
#pragma unroll
      for (int i = 0; i < C::ROWS / NW; ++i) {
        const int r = w + i * NW;
        float v[NS / 32];
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < NS / 32; ++u) {
          const int col = lane + 32 * u;
          v[u] = (base + col < count) ? Ss[r * LDS + col] : -INFINITY;
          mx = fmaxf(mx, v[u]);
        }
        mx = warp_max(mx);
        const float m_old = m_s[r];
        const float m_new = fmaxf(m_old, mx);
        float alpha = 1.f, psum = 0.f;
        if (m_new != -INFINITY) alpha = exp2f(m_old - m_new);
#pragma unroll
        for (int u = 0; u < NS / 32; ++u) {
          const float p = (m_new != -INFINITY) ? exp2f(v[u] - m_new) : 0.f;
          psum += p;
          Ps[r * LDP + lane + 32 * u] = __float2bfloat16_rn(p);
        }
        psum = warp_sum(psum);
        __syncwarp();
        if (lane == 0) {
          m_s[r] = m_new;
          l_s[r] = l_s[r] * alpha + psum;
          a_s[r] = alpha;
        }
      }
    }
    __syncthreads();
    // ---- O = O*alpha + P V -------------------------------------------------
    {
      const int mt = w % MT, cg = w / MT;
      const int cbase = cg * (D / 4);
      const float al0 = a_s[mt * 16 + g], al1 = a_s[mt * 16 + g + 8];
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        oacc[n][0] *= al0;
        oacc[n][1] *= al0;
        oacc[n][2] *= al1;
        oacc[n][3] *= al1;
      }
#pragma unroll
      for (int k = 0; k < NS / 16; ++k) {
        uint32_t a[4];
        ldsm_x4(a, Ps + (mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDP + k * 16 +
                       8 * (lane >> 4));
#pragma unroll
        for (int n2 = 0; n2 < NO; n2 += 2) {
          uint32_t bb[4];
          ldsm_x4_t(bb, KT + (k * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDQ + cbase +
                            n2 * 8 + 8 * (lane >> 4));
          mma_bf16(oacc[n2], a, bb[0], bb[1]);
          mma_bf16(oacc[n2 + 1], a, bb[2], bb[3]);
        }
      }
    }
  }
  // ---- epilogue ------------------------------------------------------------
  {
    const int mt = w % MT, cg = w / MT;
    const int cbase = cg * (D / 4);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = mt * 16 + g + 8 * half;
      const int h = h0 + r;
      if (h >= H) continue;
      const float l = l_s[r];
      const float inv = 1.f / l;
      __nv_bfloat16* orow = o + (((long long)bi * sq + t) * H + h) * D + cbase;
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        *reinterpret_cast<uint32_t*>(orow + n * 8 + 2 * cq) =
            pack_bf16(oacc[n][2 * half] * inv, oacc[n][2 * half + 1] * inv);
      }
      if (cg == 0 && cq == 0) lse[((long long)bi * sq + t) * H + h] = (m_s[r] + log2f(l)) * kLn2;
    }
  }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

// S = Q K^T and dP = dO V^T for 16 head rows (m-tile mt) x NQ*8 slots from n0,
// sharing the KV fragments (K = V).
template <int D, int NQ, int LDQ>
__device__ __forceinline__ void score_dp_tile(float (&sacc)[NQ][4], float (&pacc)[NQ][4],
                                              const __nv_bfloat16* Qs,
                                              const __nv_bfloat16* dOs,
                                              const __nv_bfloat16* KT, int mt, int n0, int lane) {
#pragma unroll
  for (int n = 0; n < NQ; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc[n][e] = pacc[n][e] = 0.f;
#pragma unroll 4
  for (int k = 0; k < D / 16; ++k) {
    uint32_t aq[4], ag[4];
    const int arow = (mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDQ + k * 16 +
                     8 * (lane >> 4);
    ldsm_x4(aq, Qs + arow);
    ldsm_x4(ag, dOs + arow);
    if constexpr (NQ == 2) {
      uint32_t bb[4];
      ldsm_x4(bb, KT + (n0 + (lane & 7) + 8 * (lane >> 4)) * LDQ + k * 16 +
                      8 * ((lane >> 3) & 1));
      mma_bf16(sacc[0], aq, bb[0], bb[1]);
      mma_bf16(sacc[1], aq, bb[2], bb[3]);
      mma_bf16(pacc[0], ag, bb[0], bb[1]);
      mma_bf16(pacc[1], ag, bb[2], bb[3]);
    } else {
      uint32_t bb[2];
      ldsm_x2(bb, KT + (n0 + (lane & 7)) * LDQ + k * 16 + 8 * ((lane >> 3) & 1));
      mma_bf16(sacc[0], aq, bb[0], bb[1]);
      mma_bf16(pacc[0], ag, bb[0], bb[1]);
    }
  }
}

// Store x0, x1 as bf16 hi parts and bf16 residuals (x - hi).
__device__ __forceinline__ void store_hi_lo(__nv_bfloat16* hi, __nv_bfloat16* lo, float x0,
                                            float x1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  *reinterpret_cast<__nv_bfloat162*>(hi) = h;
  *reinterpret_cast<__nv_bfloat162*>(lo) = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
}
template <int D, int MT>
struct BwdCfg {
  static constexpr int NW = 4 * MT;
  static constexpr int NT = NW * 32;
  static constexpr int NS = D <= 128 ? 64 : 32;
  static constexpr int ROWS = 16 * MT;
  static constexpr int LDQ = D + 8;
  static constexpr int LDP = NS + 8;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + ROWS * LDQ * 2;
  static constexpr int OFF_KV = OFF_DO + ROWS * LDQ * 2;
  static constexpr int OFF_P = OFF_KV + 2 * NS * LDQ * 2;     // P hi, P lo
  static constexpr int OFF_DS = OFF_P + 2 * ROWS * LDP * 2;   // dS hi, dS lo
  static constexpr int OFF_STAT = OFF_DS + 2 * ROWS * LDP * 2;   // lse2, D, D partials [4]
  static constexpr int OFF_ROWS = OFF_STAT + 6 * ROWS * 4;
  // dKV phase: warps split (slot m16-tile, column group)
  static constexpr int NST = NS / 16;
  static constexpr int NCG = NW / NST;
  static constexpr int NK = D / NCG / 8;
};

template <int D, int MT>
__global__ void __launch_bounds__(BwdCfg<D, MT>::NT) attn_bwd_mma(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
    const int32_t* __restrict__ idx, const float* __restrict__ sink, float scale,
    const __nv_bfloat16* __restrict__ o, const float* __restrict__ lse,
    const __nv_bfloat16* __restrict__ dO, float* __restrict__ dq, float* __restrict__ dkv,
    float* __restrict__ dsink, int sq, int H, int n_c, int ratio, int window, int K,
    const int32_t* __restrict__ doc, int tb) {
  using C = BwdCfg<D, MT>;
  constexpr int NS = C::NS, LDQ = C::LDQ, LDP = C::LDP, NT = C::NT;
  constexpr int NQ = NS / 32;
  constexpr int NO = D / 32;
  constexpr int NK = C::NK;
  static_assert(NK % 2 == 0 && NO % 2 == 0, "tile split");
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_Q);
  __nv_bfloat16* dOs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_DO);
  __nv_bfloat16* KVs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_KV);
  __nv_bfloat16* Ps = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_P);      // hi
  __nv_bfloat16* Pl = Ps + C::ROWS * LDP;                                       // lo
  __nv_bfloat16* dSs = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_DS);    // hi
  __nv_bfloat16* dSl = dSs + C::ROWS * LDP;                                     // lo
  float* lse2_s = reinterpret_cast<float*>(smem + C::OFF_STAT);
  float* D_s = lse2_s + C::ROWS;
  int* rows = reinterpret_cast<int*>(smem + C::OFF_ROWS);
  __shared__ int s_count;

  const int t = tb + (int)blockIdx.x, bi = blockIdx.y, h0 = blockIdx.z * C::ROWS;
  const int tid = threadIdx.x, w = tid / 32, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  const int n_kv = sq + n_c;
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * D;
  float* dkv_b = dkv + (long long)bi * n_kv * D;
  const long long qrow = ((long long)bi * sq + t) * H;

  if (w == 0) {
    const int c = build_slots_warp(rows, idx ? idx + ((long long)bi * sq + t) * K : nullptr, K, t,
                                   sq, n_c, ratio, window, doc ? doc + (long long)bi * sq : nullptr);
    if (lane == 0) s_count = c;
  }
  load_heads<D, C::ROWS, LDQ, NT>(Qs, q + qrow * D, h0, H);
  load_heads<D, C::ROWS, LDQ, NT>(dOs, dO + qrow * D, h0, H);
  for (int r = tid; r < C::ROWS; r += NT) {
    const int h = h0 + r;
    lse2_s[r] = (h < H) ? lse[qrow + h] * kLog2e : INFINITY;   // padded rows: p = 0
  }
  __syncthreads();
  const int count = s_count;
  const int ntiles = (count + NS - 1) / NS;
  const float sc2 = scale * kLog2e;
  const int mt_s = w % MT, grp = w / MT;

  // ---- pass 1: D_h = sum_i p_i dP_i --------------------------------------------
  {
    float dpart[2] = {0.f, 0.f};
    gather_tile<D, NS, LDQ, NT>(KVs, kv_b, rows, 0, count);
    cp_async_commit();
    for (int it = 0; it < ntiles; ++it) {
      cp_async_wait_all();
      __syncthreads();
      if (it + 1 < ntiles) {
        gather_tile<D, NS, LDQ, NT>(KVs + ((it + 1) & 1) * NS * LDQ, kv_b, rows, (it + 1) * NS,
                                    count);
        cp_async_commit();
      }
      const __nv_bfloat16* KT = KVs + (it & 1) * NS * LDQ;
      float sacc[NQ][4], pacc[NQ][4];
      score_dp_tile<D, NQ, LDQ>(sacc, pacc, Qs, dOs, KT, mt_s, grp * (NS / 4), lane);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float l2 = lse2_s[mt_s * 16 + g + 8 * half];
#pragma unroll
        for (int n = 0; n < NQ; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = grp * (NS / 4) + n * 8 + 2 * cq + e;
            if (it * NS + col < count)
              dpart[half] += exp2f(sacc[n][2 * half + e] * sc2 - l2) * pacc[n][2 * half + e];
          }
      }
    }
    // fixed-order reduction (quad lanes, then the four slot groups), so that
    // D and everything derived from it are reproducible run to run
    float* D_part = D_s + C::ROWS;   // [4][ROWS]
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v = dpart[half];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (cq == 0) D_part[grp * C::ROWS + mt_s * 16 + g + 8 * half] = v;
    }
    __syncthreads();
    for (int r = tid; r < C::ROWS; r += NT)
      D_s[r] = (D_part[r] + D_part[C::ROWS + r]) + (D_part[2 * C::ROWS + r] + D_part[3 * C::ROWS + r]);
    __syncthreads();
    // sink gradient: dsink_h = -exp(sink_h - lse) D_h
    if (sink != nullptr) {
      for (int r = tid; r < C::ROWS; r += NT) {
        const int h = h0 + r;
        if (h < H) atomicAdd(&dsink[h], -exp2f(sink[h] * kLog2e - lse2_s[r]) * D_s[r]);
      }
    }
  }

  gather_tile<D, NS, LDQ, NT>(KVs, kv_b, rows, 0, count);
  cp_async_commit();

  float dqacc[NO][4];
#pragma unroll
  for (int n = 0; n < NO; ++n) dqacc[n][0] = dqacc[n][1] = dqacc[n][2] = dqacc[n][3] = 0.f;

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait_all();
    __syncthreads();
    if (it + 1 < ntiles) {
      gather_tile<D, NS, LDQ, NT>(KVs + ((it + 1) & 1) * NS * LDQ, kv_b, rows, (it + 1) * NS,
                                  count);
      cp_async_commit();
    }
    const __nv_bfloat16* KT = KVs + (it & 1) * NS * LDQ;
    const int base = it * NS;
    // ---- S = Q K^T, dP = dO V^T; P and dS (hi, lo) to smem ------------------
    {
      float sacc[NQ][4], pacc[NQ][4];
      const int n0 = grp * (NS / 4);
      score_dp_tile<D, NQ, LDQ>(sacc, pacc, Qs, dOs, KT, mt_s, n0, lane);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = mt_s * 16 + g + 8 * half;
        const float l2 = lse2_s[r], Dh = D_s[r];
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
          const int col = n0 + n * 8 + 2 * cq;
          float pv[2], dv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool ok = base + col + e < count;
            const float p = ok ? exp2f(sacc[n][2 * half + e] * sc2 - l2) : 0.f;
            pv[e] = p;
            dv[e] = p * (pacc[n][2 * half + e] - Dh) * scale;
          }
          store_hi_lo(Ps + r * LDP + col, Pl + r * LDP + col, pv[0], pv[1]);
          store_hi_lo(dSs + r * LDP + col, dSl + r * LDP + col, dv[0], dv[1]);
        }
      }
    }
    __syncthreads();
    // ---- dQ += dS K ----------------------------------------------------------
    {
      const int mt = w % MT, cg = w / MT;
      const int cbase = cg * (D / 4);
#pragma unroll
      for (int k = 0; k < NS / 16; ++k) {
        uint32_t a[4], al[4];
        const int aoff = (mt * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDP + k * 16 +
                         8 * (lane >> 4);
        ldsm_x4(a, dSs + aoff);
        ldsm_x4(al, dSl + aoff);
#pragma unroll
        for (int n2 = 0; n2 < NO; n2 += 2) {
          uint32_t bb[4];
          ldsm_x4_t(bb, KT + (k * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDQ + cbase +
                            n2 * 8 + 8 * (lane >> 4));
          mma_bf16(dqacc[n2], a, bb[0], bb[1]);
          mma_bf16(dqacc[n2 + 1], a, bb[2], bb[3]);
          mma_bf16(dqacc[n2], al, bb[0], bb[1]);
          mma_bf16(dqacc[n2 + 1], al, bb[2], bb[3]);
        }
      }
    }
    // ---- dKV_tile = P^T dO + dS^T Q, scattered with fp32 atomics -------------
    {
      const int st = w % C::NST, cg = w / C::NST;
      const int cbase = cg * (D / C::NCG);
      float kacc[NK][4];
#pragma unroll
      for (int n = 0; n < NK; ++n) kacc[n][0] = kacc[n][1] = kacc[n][2] = kacc[n][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < MT; ++kk) {
        uint32_t ap[4], ad[4], apl[4], adl[4];
        const int aoff = (kk * 16 + (lane & 7) + 8 * (lane >> 4)) * LDP + st * 16 +
                         8 * ((lane >> 3) & 1);
        ldsm_x4_t(ap, Ps + aoff);
        ldsm_x4_t(ad, dSs + aoff);
        ldsm_x4_t(apl, Pl + aoff);
        ldsm_x4_t(adl, dSl + aoff);
#pragma unroll
        for (int n2 = 0; n2 < NK; n2 += 2) {
          const int boff = (kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * LDQ + cbase +
                           n2 * 8 + 8 * (lane >> 4);
          uint32_t bg[4], bq[4];
          ldsm_x4_t(bg, dOs + boff);
          ldsm_x4_t(bq, Qs + boff);
          mma_bf16(kacc[n2], ap, bg[0], bg[1]);
          mma_bf16(kacc[n2 + 1], ap, bg[2], bg[3]);
          mma_bf16(kacc[n2], apl, bg[0], bg[1]);
          mma_bf16(kacc[n2 + 1], apl, bg[2], bg[3]);
          mma_bf16(kacc[n2], ad, bq[0], bq[1]);
          mma_bf16(kacc[n2 + 1], ad, bq[2], bq[3]);
          mma_bf16(kacc[n2], adl, bq[0], bq[1]);
          mma_bf16(kacc[n2 + 1], adl, bq[2], bq[3]);
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int p = base + st * 16 + g + 8 * half;
        if (p < count) {
          float* drow = dkv_b + (long long)rows[p] * D + cbase + 2 * cq;
#pragma unroll
          for (int n = 0; n < NK; ++n)
            red_add_v2(drow + n * 8, kacc[n][2 * half], kacc[n][2 * half + 1]);
        }
      }
    }
  }
  // ---- dq ----------------------------------------------------------------------
  {
    const int mt = w % MT, cg = w / MT;
    const int cbase = cg * (D / 4);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int h = h0 + mt * 16 + g + 8 * half;
      if (h >= H) continue;
      float* drow = dq + (qrow + h) * D + cbase;
#pragma unroll
      for (int n = 0; n < NO; ++n)
        *reinterpret_cast<float2*>(drow + n * 8 + 2 * cq) =
            make_float2(dqacc[n][2 * half], dqacc[n][2 * half + 1]);
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <int D, int MT>
static cudaError_t run_fwd(const void* q, const void* kv, const int32_t* idx, const float* sink,
                           float scale, void* o, float* lse, int b, int sq, int H, int n_c,
                           int ratio, int window, int K, cudaStream_t s, const int32_t* doc,
                           int tb, int te) {
  using C = FwdCfg<D, MT>;
  const size_t smem = C::OFF_ROWS + (size_t)(window + (idx ? K : n_c) + 32) * sizeof(int);
  auto k = attn_fwd_mma<D, MT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(te - tb), (unsigned)b, (unsigned)((H + C::ROWS - 1) / C::ROWS));
  k<<<grid, C::NT, smem, s>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx, sink, scale,
                              (__nv_bfloat16*)o, lse, sq, H, n_c, ratio, window, K, doc, tb);
    count_launches(1);
  return cudaGetLastError();
}

template <int D, int MT>
static cudaError_t run_bwd(const void* q, const void* kv, const int32_t* idx, const float* sink,
                           float scale, const void* o, const float* lse, const void* dO, float* dq,
                           float* dkv, float* dsink, int b, int sq, int H, int n_c, int ratio,
                           int window, int K, cudaStream_t s, const int32_t* doc, int tb,
                           int te) {
  using C = BwdCfg<D, MT>;
  const size_t smem = C::OFF_ROWS + (size_t)(window + (idx ? K : n_c) + 32) * sizeof(int);
  auto k = attn_bwd_mma<D, MT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(te - tb), (unsigned)b, (unsigned)((H + C::ROWS - 1) / C::ROWS));
  k<<<grid, C::NT, smem, s>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx, sink, scale,
                              (const __nv_bfloat16*)o, lse, (const __nv_bfloat16*)dO, dq, dkv,
                              dsink, sq, H, n_c, ratio, window, K, doc, tb);
    count_launches(1);
  return cudaGetLastError();
}

// Tensor-core path available for this shape?  (bf16, d in {64,128,256,512},
// smem for the slot list within budget.)
bool attn_mma_supported(int H, int d, int window, int K) {
  (void)H;
  if (!(d == 64 || d == 128 || d == 256 || d == 512)) return false;
  return (size_t)(window + K) * 4 < 16 * 1024;
}

cudaError_t launch_attn_fwd_mma(const void* q, const void* kv, const int32_t* idx,
                                const float* sink, float scale, void* o, float* lse, int b, int sq,
                                int H, int d, int n_c, int ratio, int window, int K,
                                cudaStream_t s, const int32_t* doc, int tb, int te) {
  const int mt = (H + 15) / 16;
#define CSA_FWD(DD, MM)                                                                      \
  return run_fwd<DD, MM>(q, kv, idx, sink, scale, o, lse, b, sq, H, n_c, ratio, window, K, s, \
                         doc, tb, te)
  switch (d) {
    case 64:
      if (mt <= 1) CSA_FWD(64, 1);
      if (mt <= 2) CSA_FWD(64, 2);
      CSA_FWD(64, 4);
    case 128:
      if (mt <= 1) CSA_FWD(128, 1);
      if (mt <= 2) CSA_FWD(128, 2);
      CSA_FWD(128, 4);
    case 256:
      if (mt <= 2) CSA_FWD(256, 2);
      CSA_FWD(256, 4);
    default:
      if (mt <= 2) CSA_FWD(512, 2);
      CSA_FWD(512, 4);
  }
#undef CSA_FWD
}

cudaError_t launch_attn_bwd_mma(const void* q, const void* kv, const int32_t* idx,
                                const float* sink, float scale, const void* o, const float* lse,
                                const void* dO, float* dq, float* dkv, float* dsink, int b, int sq,
                                int H, int d, int n_c, int ratio, int window, int K,
                                cudaStream_t s, const int32_t* doc, int tb, int te) {
  const int mt = (H + 15) / 16;
#define CSA_BWD(DD, MM)                                                                       \
  return run_bwd<DD, MM>(q, kv, idx, sink, scale, o, lse, dO, dq, dkv, dsink, b, sq, H, n_c, \
                         ratio, window, K, s, doc, tb, te)
  switch (d) {
    case 64:
      if (mt <= 1) CSA_BWD(64, 1);
      if (mt <= 2) CSA_BWD(64, 2);
      CSA_BWD(64, 4);
    case 128:
      if (mt <= 1) CSA_BWD(128, 1);
      if (mt <= 2) CSA_BWD(128, 2);
      CSA_BWD(128, 4);
    case 256:
      CSA_BWD(256, 2);
    default:
      CSA_BWD(512, 2);
  }
#undef CSA_BWD
}

}  // namespace csa
