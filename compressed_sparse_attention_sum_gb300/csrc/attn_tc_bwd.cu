// Sparse MQA backward on the 5th-generation tensor cores (tcgen05 + TMEM),
// bf16, d = 128.
//
// Semantics as csa_attn_bwd ("Add unfused SBHD compressed sparse attention",
// review of the gather backward: compact [b*n_kv, d] dKV with repeated
// indices summed; "Add the min-memory DSA attention kernels": fp32 scatter):
//   D = sum_i p_i dP_i,  p_i = exp(s_i - lse),  ds_i = p_i (dP_i - D),
//   dq = scale sum_i ds_i kv_i,  dkv_i += p_i dO + scale ds_i q,
//   dsink = -exp(sink - lse) D.
//
// The CTA owns the same 128 (query, head) rows and walks the same union of
// slots as the tensor-core forward.  TMEM holds four 128-column fp32 blocks:
// S (rows x slots), dP (rows x slots), the tile's dKV (slots x d) and the
// running dQ (rows x d).  Pass 1 forms D = sum p dP per row exactly (the
// bf16 rounding of the stored O would move dq and dkv by up to 1e-2 when a
// query has few slots); during pass 1 the dKV/dQ columns are free, so S and dP
// alternate between two TMEM buffers and the next tile's MMAs overlap this
// tile's sum.  Pass 2, per tile of 128 slots:
//   S = Q K^T, dP = dO V^T                       (K-major A and B)
//   P as bf16 hi + lo -> smem X, Y;  dKV = P^T dO   (A = P^T and B = dO read
//                                                  MN-major from the same tiles)
//   dS*scale (computed while the tensor core forms P^T dO) as bf16 hi + lo
//   -> X, Y; dKV += dS^T Q; dQ += dS K
//   dKV (summed over the block's heads and queries inside the MMA) is
//   scattered into the compact buffer with fp32 vector atomics.
// The hi/lo split carries ~16 significant bits of P and dS into the
// products, so the fp32 sums over thousands of queries stay accurate.
// KV tiles are double-buffered: the next tile's gather overlaps this tile.
// The CTAs are persistent (one per SM) and walk the query blocks heaviest
// first; the next block's Q and dO tiles are requested as soon as the last
// products of the current block have read them.
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"
#include "attn_union.cuh"

#include <cudaTypedefs.h>

namespace csa {
namespace atb {

using namespace csa::umma;

constexpr int kRows = 128;
constexpr int kSlots = 128;
constexpr int kD = 128;
constexpr int kThreads = 512;                   // 16 warps: TMEM lane quarter x column quarter
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDKV = 256, kColDQ = 384;
constexpr uint32_t kBlk = kRows * 128;          // 16 KB: 128 lines of 128 B

struct Layout {
  static constexpr uint32_t Q = 0;              // [2][128][128 B] K-major
  static constexpr uint32_t DO = 2 * kBlk;
  static constexpr uint32_t KV = 4 * kBlk;      // two buffers of 2 blocks
  static constexpr uint32_t X = 8 * kBlk;       // P / dS hi
  static constexpr uint32_t Y = 10 * kBlk;      // P / dS lo
  static constexpr uint32_t BARS = 12 * kBlk;   // q, sp, p, ds, pass-1 buffers 0/1
  static constexpr uint32_t TSLOT = BARS + 6 * 8;
  static constexpr uint32_t SCAL = TSLOT + 8;
  static constexpr uint32_t RED = SCAL + 64;    // [4][128] floats
  static constexpr uint32_t CONTRIB = RED + 2048;   // [128] floats
  static constexpr uint32_t BIAS = CONTRIB + 512;   // [2][QB][128] floats
};

__device__ __forceinline__ uint32_t sw_off(int r, int ch) {
  return (uint32_t)((ch >> 3) * kBlk + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async_commit_() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group_() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Store two halves of 8 values as bf16 hi (to X) and bf16 residual (to Y).
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

template <int QB>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_do,
    const __nv_bfloat16* __restrict__ kv, const __nv_bfloat16* __restrict__ dO_g,
    const int32_t* __restrict__ idx,
    const float* __restrict__ sink, float scale, const __nv_bfloat16* __restrict__ o,
    const float* __restrict__ lse, float* __restrict__ dq, float* __restrict__ dkv, float* __restrict__ dsink, int sq, int H,
    int n_c, int ratio, int window, int K, int* __restrict__ status,
    const int32_t* __restrict__ doc, int tb, int te, int njobs) {
  constexpr int NW = (QB + 3) / 4;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + Layout::BARS);
  uint64_t* bar_sp = bar_q + 1;
  uint64_t* bar_p = bar_q + 2;
  uint64_t* bar_ds = bar_q + 3;
  uint64_t* bar_d1 = bar_q + 4;          // [2] pass-1 S/dP buffers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::TSLOT);
  int* scal = reinterpret_cast<int*>(sm + Layout::SCAL);
  float* red = reinterpret_cast<float*>(sm + Layout::RED);
  float* contrib = reinterpret_cast<float*>(sm + Layout::CONTRIB);
  float* bias = reinterpret_cast<float*>(sm + Layout::BIAS);                 // [2][QB][128]
  uint64_t* cnt = reinterpret_cast<uint64_t*>(bias + 2 * QB * kSlots);       // [n_c][NW]
  int* ulist = reinterpret_cast<int*>(cnt + (size_t)n_c * NW);               // [n_c]
  int* wsum = ulist + n_c;                                                   // [16]
  unsigned char* X = sm + Layout::X;
  unsigned char* Y = sm + Layout::Y;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = (te - tb + QB - 1) / QB;
  const int nb = njobs / nblk;       // batch elements
  const int n_kv = sq + n_c;
  // Persistent CTAs: job j is query block nblk-1-j/nb of batch element j%nb
  // (the work of a block grows with its position, so the jobs run heaviest
  // first), dealt to the CTAs in sweeps of G jobs whose order alternates
  // (CTA c takes job c of sweep 0, job 2G-1-c of sweep 1, ...), which evens
  // out the CTAs' totals
  const int G = (int)gridDim.x;
  auto job_of = [&](int sweep) -> int {
    const int c = (sweep & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const int j = sweep * G + c;
    return j < njobs ? j : -1;
  };

  // ---- set-up (once per CTA): barriers, TMEM ------------------------------------
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_sp, 1);
    mbar_init(bar_p, 2);                 // P^T dO: hi and lo parts issued by two threads
    mbar_init(bar_ds, 1);
    mbar_init(bar_d1, 2);                // pass 1: S and dP issued by two threads
    mbar_init(bar_d1 + 1, 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  // Q and dO tiles of job j (issued by thread 0)
  auto load_qdo = [&](int j) {
    const int row0 = ((j % nb) * sq + tb + (nblk - 1 - j / nb) * QB) * H;
    mbar_expect_tx(bar_q, 4 * kBlk);
    tma_load_2d(sm + Layout::Q, &tmap_q, bar_q, 0, row0);
    tma_load_2d(sm + Layout::Q + kBlk, &tmap_q, bar_q, 64, row0);
    tma_load_2d(sm + Layout::DO, &tmap_do, bar_q, 0, row0);
    tma_load_2d(sm + Layout::DO + kBlk, &tmap_do, bar_q, 64, row0);
  };

  // ---- per-thread state -------------------------------------------------------
  const int qd = warp & 3, hf = warp >> 2;         // hf: column group (32 columns)
  const int r = qd * 32 + lane;                    // TMEM lane: row (S, dP, dQ) or slot (dKV)
  const int q = r / H, h = r % H;
  const float sc2 = scale * kLog2e;
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const uint32_t tS = tmem + lane_base + kColS + hf * 32;
  const uint32_t tDP = tmem + lane_base + kColDP + hf * 32;
  const uint32_t tDKV = tmem + lane_base + kColDKV + hf * 32;
  const uint32_t tDQ = tmem + lane_base + kColDQ + hf * 32;
  // completed phases of the barriers, carried across this CTA's jobs
  uint32_t n_q = 0, n_sp = 0, n_p = 0, n_ds = 0, n_d1a = 0, n_d1b = 0;
  bool ok = true;
  int site = 0;
  int job = job_of(0);
  if (tid == 0 && job >= 0) load_qdo(job);

  for (int sweep = 0; job >= 0; ++sweep) {
  const int bi = job % nb, xb = nblk - 1 - job / nb;
  const int t0 = tb + xb * QB;       // rows t0 .. t0+QB-1 below te are this block's queries
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * kD;
  float* dkv_b = dkv + (long long)bi * n_kv * kD;
  const int next = job_of(sweep + 1);

  // ---- union of the block's selected compressed blocks ----------------------
  for (int e = tid; e < n_c * NW; e += kThreads) cnt[e] = 0ull;
  __syncthreads();
  const int t_last = min(t0 + QB, te) - 1;
  const int nu = build_union<QB, kThreads>(idx, bi, sq, K, t0, te, ratio, n_c, cnt, ulist, wsum,
                                           scal);
  const int win0 = max(0, t0 - window + 1);
  const int nwin = t_last - win0 + 1;
  const int S_total = nwin + nu;
  const int ntiles = (S_total + kSlots - 1) / kSlots;

  auto slot_row = [&](int s) -> int {
    return s < nwin ? win0 + s : (s < S_total ? sq + ulist[s - nwin] : 0);
  };
  // gather tile `it` into KV buffer (it & 1) and its bias table
  auto stage_tile = [&](int it) {
    const int sbase = it * kSlots;
    unsigned char* dst = sm + Layout::KV + (it & 1) * 2 * kBlk;
    for (int c = tid; c < kSlots * 16; c += kThreads) {
      const int rr = c >> 4, ch = c & 15;
      if (sbase + rr >= S_total) {       // padding: zeros, not a shared hot row
        *reinterpret_cast<uint4*>(dst + sw_off(rr, ch)) = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      cp_async_16(dst + sw_off(rr, ch), kv_b + (long long)slot_row(sbase + rr) * kD + ch * 8);
    }
    cp_async_commit_();
    float* bt = bias + (it & 1) * QB * kSlots;
    for (int e = tid; e < QB * kSlots; e += kThreads) {
      const int qq = e / kSlots, c = e % kSlots;
      const int s = sbase + c;
      const int tq = t0 + qq;
      float bv = -INFINITY;
      if (tq < te) {
        if (s < nwin) {
          const int raw = win0 + s;
          if (raw <= tq && raw > tq - window &&
              (doc == nullptr || __ldg(doc + (long long)bi * sq + raw) == __ldg(doc + (long long)bi * sq + tq)))
            bv = 0.f;
        } else if (s < S_total) {
          const int j = ulist[s - nwin];
          const uint32_t cq = (uint32_t)(cnt[j * NW + (qq >> 2)] >> (16 * (qq & 3))) & 0xFFFFu;
          if (cq != 0u) bv = cq == 1u ? 0.f : log2f((float)cq);
        }
      }
      bt[e] = bv;
    }
  };

  // ---- this block's rows ------------------------------------------------------
  const int t = t0 + q;
  const bool row_ok = t < te;
  const float lse2 = row_ok ? lse[(long long)(bi * sq + t0) * H + r] * kLog2e : INFINITY;
  ok = __syncthreads_and(mbar_wait(bar_q, n_q & 1));
  if (!ok) { site = kSiteBwdQ; break; }
  ++n_q;

  auto issue_s_dp = [&](int it) {
    constexpr uint32_t idesc = idesc_bf16_f32_major(kRows, kSlots, 0, 0);
    const uint32_t qa = smem_addr(sm + Layout::Q), ga = smem_addr(sm + Layout::DO);
    const uint32_t ka = smem_addr(sm + Layout::KV + (it & 1) * 2 * kBlk);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k) {
      const uint32_t off = (k >> 2) * kBlk + (k & 3) * 32;
      mma_bf16_ss(tmem + kColS, sw128_desc(qa + off), sw128_desc(ka + off), idesc, k > 0);
      mma_bf16_ss(tmem + kColDP, sw128_desc(ga + off), sw128_desc(ka + off), idesc, k > 0);
    }
    mma_commit(bar_sp);
  };

  // ---- pass 1: D = sum_i p_i dP_i (S/dP double-buffered in TMEM) --------------------
  {
    // S (thread 0) and dP (thread 32) of tile `it`: tcgen05.mma holds its
    // issuing thread while the tensor core works through it, so two issuers
    // each keep their warp from its share of the sum for half as long
    auto issue_pass1 = [&](int it, bool dp) {
      constexpr uint32_t idesc = idesc_bf16_f32_major(kRows, kSlots, 0, 0);
      const uint32_t aa = smem_addr(sm + (dp ? Layout::DO : Layout::Q));
      const uint32_t ka = smem_addr(sm + Layout::KV + (it & 1) * 2 * kBlk);
      const uint32_t cs = (it & 1) * 256 + (dp ? 128 : 0);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {
        const uint32_t off = (k >> 2) * kBlk + (k & 3) * 32;
        mma_bf16_ss(tmem + cs, sw128_desc(aa + off), sw128_desc(ka + off), idesc, k > 0);
      }
      mma_commit(&bar_d1[it & 1]);
    };
    float dpart = 0.f;
    if (ok && ntiles > 0) {
      stage_tile(0);
      if (ntiles > 1) {
        stage_tile(1);
        cp_async_wait_group_<1>();
      } else {
        cp_async_wait_group_<0>();
      }
      fence_proxy_async_smem();
      fence_before();
      __syncthreads();
      if (tid == 0 || tid == 32) {
        fence_after();
        issue_pass1(0, tid == 32);
      }
    }
    for (int it = 0; it < ntiles && ok; ++it) {
      if (it + 1 < ntiles) {
        // tile it+1 is staged: start its MMAs into the other TMEM buffer
        cp_async_wait_group_<0>();
        fence_proxy_async_smem();
        fence_before();
        __syncthreads();
        if (tid == 0 || tid == 32) {
          fence_after();
          issue_pass1(it + 1, tid == 32);
        }
      }
      // per-warp wait: a warp sums as soon as the products are there, not
      // after the two issuing threads have handed the next tile's over (the
      // barrier below carries a failed wait to every thread)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&bar_d1[it & 1], (((it & 1) ? n_d1b : n_d1a) + (it >> 1)) & 1));
      if (ok) {
        fence_after();
        const float* bq = bias + (it & 1) * QB * kSlots + q * kSlots + hf * 32;
        const uint32_t cs = lane_base + (it & 1) * 256 + hf * 32;
        uint32_t vs[32], vp[32];
        CSA_TMEM_LD32(tmem + cs, vs);
        CSA_TMEM_LD32(tmem + cs + 128, vp);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        CSA_TMEM_WAIT32(vs);
        CSA_TMEM_WAIT32(vp);
#pragma unroll
        for (int c = 0; c < 32; ++c)
          dpart = fmaf(ex2(fmaf(__uint_as_float(vs[c]), sc2, bq[c] - lse2)),
                       __uint_as_float(vp[c]), dpart);
      }
      fence_before();
      // everyone is done with this tile's bias table and TMEM buffer; its KV
      // buffer was released when its MMAs completed: stage tile it+2 there
      ok = __syncthreads_and(ok);
      if (!ok) { site = kSiteBwdS; break; }
      if (it + 2 < ntiles) stage_tile(it + 2);
    }
    red[hf * kRows + r] = dpart;
    n_d1a += (ntiles + 1) / 2;
    n_d1b += ntiles / 2;
  }
  if (!ok) break;
  // the tile's dKV accumulator starts from zero: every MMA into it accumulates,
  // so that its hi and lo parts may be issued by two threads in any order
  {
    uint32_t z[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) z[c] = 0u;
    CSA_TMEM_ST32(tDKV, z);
    tmem_wait_st();
  }
  fence_before();
  __syncthreads();
  const float Drow = (red[r] + red[kRows + r]) + (red[2 * kRows + r] + red[3 * kRows + r]);

  // ---- pass 2 ---------------------------------------------------------------------
  // Tiles in descending order: pass 1 left its last two tiles (and their bias
  // tables) in the two KV buffers, so the first two need no gather (the
  // barrier above ordered every read of pass 1's TMEM before this issue).
  if (ok && ntiles > 0 && tid == 0) {
    fence_after();
    bulk_wait_read_all();      // the previous block's dq copy has read X|Y
    issue_s_dp(ntiles - 1);
  }
  for (int it = 0; it < ntiles && ok; ++it) {
    const int tt = ntiles - 1 - it;    // the tile of this iteration
    // the gather of tile tt-1 overlaps this tile (the buffer of tile tt+1 was
    // released when that tile's MMAs completed); tile ntiles-2 is resident
    if (it > 0 && tt > 0) stage_tile(tt - 1);
    ok = __syncthreads_and(mbar_wait(bar_sp, n_sp & 1));
    ++n_sp;
    if (!ok) { site = kSiteBwdS; break; }
    fence_after();
    const float* bq = bias + (tt & 1) * QB * kSlots + q * kSlots + hf * 32;
    // P (hi, lo) -> X, Y
    {
      uint32_t vs[32];
      tmem_ld32_wait(tS, vs);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = ex2(fmaf(__uint_as_float(vs[c8 * 8 + e]), sc2, bq[c8 * 8 + e] - lse2));
          vs[c8 * 8 + e] = __float_as_uint(p[e]);
        }
        store_hi_lo8(X, Y, sw_off(r, hf * 4 + c8), p);
      }
      // keep P (fp32) in the S columns for the dS step
      CSA_TMEM_ST32(tS, vs);
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0 || tid == 32) {
      fence_after();
      // dKV += P^T dO: M = slots, N = d, K = rows; A = P^T (MN-major view of
      // X for the hi part, issued by thread 0, and of Y for the lo part,
      // thread 32), B = dO (MN-major view of its K-major tile)
      constexpr uint32_t idesc = idesc_bf16_f32_major(kSlots, kD, 1, 1);
      const uint32_t pa = smem_addr(tid == 0 ? X : Y), ga = smem_addr(sm + Layout::DO);
#pragma unroll
      for (int k = 0; k < kRows / 16; ++k)
        mma_bf16_ss(tmem + kColDKV, sw128_desc_mn(pa + k * 2048, kBlk),
                    sw128_desc_mn(ga + k * 2048, kBlk), idesc, 1u);
      mma_commit(bar_p);
    }
    // dS * scale from P (kept in the S columns) and dP while the tensor core
    // works on P^T dO; it goes to X, Y once that product has read them
    float dsv[32];
    {
      uint32_t vs[32], vp[32];
      CSA_TMEM_LD32(tS, vs);
      CSA_TMEM_LD32(tDP, vp);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      CSA_TMEM_WAIT32(vs);
      CSA_TMEM_WAIT32(vp);
#pragma unroll
      for (int c = 0; c < 32; ++c)
        dsv[c] = __uint_as_float(vs[c]) * (__uint_as_float(vp[c]) - Drow) * scale;
    }
    ok = __syncthreads_and(mbar_wait(bar_p, n_p & 1));
    ++n_p;
    if (!ok) { site = kSiteBwdP; break; }
    fence_after();
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8)
      store_hi_lo8(X, Y, sw_off(r, hf * 4 + c8),
                   *reinterpret_cast<const float(*)[8]>(dsv + c8 * 8));
    if (it > 0 && tt > 0) cp_async_wait_group_<0>();
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0) {
      fence_after();
      const uint32_t xa = smem_addr(X), ya = smem_addr(Y);
      const uint32_t qa = smem_addr(sm + Layout::Q);
      const uint32_t ka = smem_addr(sm + Layout::KV + (tt & 1) * 2 * kBlk);
      // dKV += dS^T Q
      constexpr uint32_t idesc_kv = idesc_bf16_f32_major(kSlots, kD, 1, 1);
#pragma unroll
      for (int k = 0; k < kRows / 16; ++k) {
        const uint64_t b = sw128_desc_mn(qa + k * 2048, kBlk);
        mma_bf16_ss(tmem + kColDKV, sw128_desc_mn(xa + k * 2048, kBlk), b, idesc_kv, 1u);
        mma_bf16_ss(tmem + kColDKV, sw128_desc_mn(ya + k * 2048, kBlk), b, idesc_kv, 1u);
      }
      // dQ += dS K: M = rows, N = d, K = slots; A = dS (K-major X/Y), B = KV (MN-major)
      constexpr uint32_t idesc_q = idesc_bf16_f32_major(kRows, kD, 0, 1);
#pragma unroll
      for (int k = 0; k < kSlots / 16; ++k) {
        const uint32_t aoff = (k >> 2) * kBlk + (k & 3) * 32;
        const uint64_t b = sw128_desc_mn(ka + k * 2048, kBlk);
        mma_bf16_ss(tmem + kColDQ, sw128_desc(xa + aoff), b, idesc_q, (it > 0 || k > 0) ? 1u : 0u);
        mma_bf16_ss(tmem + kColDQ, sw128_desc(ya + aoff), b, idesc_q, 1u);
      }
      mma_commit(bar_ds);
    }
    ok = __syncthreads_and(mbar_wait(bar_ds, n_ds & 1));
    ++n_ds;
    if (!ok) { site = kSiteBwdDS; break; }
    fence_after();
    // scatter this tile's dKV rows (TMEM lane = slot) into the compact buffer,
    // while the tensor core computes the next tile's S and dP: stage the fp32
    // rows contiguously in X|Y (free until the next tile's P), then one
    // coalesced fp32 vector reduction of 512 B per valid slot row
    {
      float* stg = reinterpret_cast<float*>(X);          // [128 slots][128] fp32 = 64 KB
      uint32_t v[32];
      tmem_ld32_wait(tDKV, v);
      {  // the next tile's dKV accumulates from zero
        uint32_t z[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) z[c] = 0u;
        CSA_TMEM_ST32(tDKV, z);
        tmem_wait_st();
      }
      float* srow = stg + r * kD + hf * 32;
      // Store chunk (c + lane) % 8 at step c so that the 32 lanes (32 rows,
      // 512 B apart) hit different banks: rotate the eight 4-float chunks by
      // lane % 8 with a 3-stage barrel shift (static register indices only).
      float4 ch[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        ch[c] = make_float4(__uint_as_float(v[c * 4]), __uint_as_float(v[c * 4 + 1]),
                            __uint_as_float(v[c * 4 + 2]), __uint_as_float(v[c * 4 + 3]));
#pragma unroll
      for (int k = 1; k < 8; k <<= 1) {
        const bool rot = (lane & k) != 0;
        float4 tmp[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) tmp[c] = rot ? ch[(c + k) & 7] : ch[c];
#pragma unroll
        for (int c = 0; c < 8; ++c) ch[c] = tmp[c];
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(srow + ((c + lane) & 7) * 4) = ch[c];
      __syncthreads();
      // S and dP of the next tile (S/dP were fully read before the dS MMAs;
      // its KV rows arrived before them): thread 0 issues them here, so that
      // the issue, which blocks while the MMA queue drains, overlaps the
      // reductions of the other warps instead of delaying everyone
      if (tid == 0 && tt > 0) {
        fence_after();
        issue_s_dp(tt - 1);
      }
      // warps 1..15, one staged row each at a time: its 32 lanes add the
      // row's 512 B with one coalesced vector reduction (X|Y is free again
      // once every thread has passed the next barrier)
      const int nrow = min(kSlots, S_total - tt * kSlots);
#pragma unroll 4
      for (int rr = warp - 1; warp > 0 && rr < nrow; rr += kThreads / 32 - 1) {
        const float4 v4 = *reinterpret_cast<const float4*>(stg + rr * kD + lane * 4);
        red_add_v4(dkv_b + (long long)slot_row(tt * kSlots + rr) * kD + lane * 4, v4.x, v4.y,
                   v4.z, v4.w);
      }
    }
    fence_before();
  }
  if (!ok) break;
  // the next job's Q and dO tiles (this block's last products, which read
  // them, have completed) stream in under this block's last reductions and
  // epilogue
  if (tid == 0 && next >= 0) load_qdo(next);
  // ---- sink gradient: -exp(sink - lse) D, summed over the block's queries per head --
  if (hf == 0)
    contrib[r] = (row_ok && sink != nullptr) ? -exp2f(sink[h] * kLog2e - lse2) * Drow : 0.f;
  __syncthreads();
  if (sink != nullptr && tid < H) {
    float sacc = 0.f;
    for (int qq = 0; qq < QB; ++qq) sacc += contrib[qq * H + tid];
    atomicAdd(&dsink[tid], sacc);
  }
  // ---- dq rows: staged in X|Y (the last drain has read its rows), then one
  // bulk copy of the block's contiguous rows, so that no warp waits for the
  // stores behind the last reductions; X|Y is next written in the next
  // block's pass 2, after the copy has read it -----------------------------------
  if (ntiles > 0) {
    uint32_t v[32];
    tmem_ld32_wait(tDQ, v);
    float* srow = reinterpret_cast<float*>(X) + r * kD + hf * 32;
    // chunk (c + lane) % 8 at step c: the 32 rows, 512 B apart, hit
    // different banks (the drain's rotation)
    float4 ch[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      ch[c] = make_float4(__uint_as_float(v[c * 4]), __uint_as_float(v[c * 4 + 1]),
                          __uint_as_float(v[c * 4 + 2]), __uint_as_float(v[c * 4 + 3]));
#pragma unroll
    for (int k = 1; k < 8; k <<= 1) {
      const bool rot = (lane & k) != 0;
      float4 tmp[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) tmp[c] = rot ? ch[(c + k) & 7] : ch[c];
#pragma unroll
      for (int c = 0; c < 8; ++c) ch[c] = tmp[c];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<float4*>(srow + ((c + lane) & 7) * 4) = ch[c];
    fence_proxy_async_smem();
  }
  // this block's TMEM and shared-memory reads are done before the next block
  fence_before();
  __syncthreads();
  if (tid == 0 && ntiles > 0) {
    const int nrows = min(QB, te - t0) * H;
    bulk_store(dq + (long long)(bi * sq + t0) * H * kD, X, (uint32_t)nrows * kD * 4u);
    bulk_commit();
  }
  job = next;
  }  // jobs

  cp_async_wait_all_();                               // no copy in flight past this point
  if (tid == 0) bulk_wait_all();                       // nor a dq copy
  // a failed wait for the prefetched tiles may leave them in flight (every
  // other wait precedes the next prefetch): wait for them once more (bounded)
  if (site == kSiteBwdQ && tid == 0) mbar_wait(bar_q, n_q & 1);
  if (!ok && tid == 0) set_status(status, kDevTimeout, site);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace atb

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_bwd() {
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

size_t attn_tc_bwd_smem(int QB, int n_c) {
  const int NW = (QB + 3) / 4;
  return 1024 + atb::Layout::BIAS + (size_t)2 * QB * atb::kSlots * 4 + (size_t)n_c * NW * 8 +
         (size_t)n_c * 4 + 64;
}

bool make_rows_map(CUtensorMap* m, const void* base, long long rows) {
  auto encode = encode_fn_bwd();
  if (encode == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)atb::kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)atb::kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)atb::kRows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}
}  // namespace

bool attn_tc_bwd_supported(int H, int d, int n_c, int K) {
  if (d != 128 || !(H == 16 || H == 32 || H == 64) || K > 65535) return false;
  if (encode_fn_bwd() == nullptr) return false;
  return attn_tc_bwd_smem(128 / H, n_c) <= 227 * 1024;
}

cudaError_t launch_attn_bwd_tc(const void* q, const void* kv, const int32_t* idx,
                               const float* sink, float scale, const void* o, const float* lse,
                               const void* dO,
                               float* dq, float* dkv, float* dsink, int b, int sq, int H, int n_c,
                               int ratio, int window, int K, int* status, cudaStream_t s,
                               const int32_t* doc, int tb, int te) {
  CUtensorMap tq, tg;
  const long long rows = (long long)b * sq * H;
  if (!make_rows_map(&tq, q, rows) || !make_rows_map(&tg, dO, rows)) return cudaErrorInvalidValue;
  const int QB = 128 / H;
  const size_t smem = attn_tc_bwd_smem(QB, n_c);
  const int njobs = ((te - tb + QB - 1) / QB) * b;
  int dev = 0, n_sm = 0;                                   // persistent CTAs: one per SM
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1)
    return cudaErrorInvalidValue;
  // With packed documents the work of a block restarts at every document,
  // so the alternating deal of the heaviest-first order does not balance the
  // CTAs: one CTA per job then (the hardware places them as SMs free up).
  const int ncta = doc != nullptr ? njobs : (njobs < n_sm ? njobs : n_sm);
  dim3 grid((unsigned)ncta);
#define CSA_TC_BWD(QQ)                                                                        \
  {                                                                                           \
    auto k = atb::attn_bwd_tc_kernel<QQ>;                                                     \
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);         \
    k<<<grid, atb::kThreads, smem, s>>>(tq, tg, (const __nv_bfloat16*)kv,                   \
                                        (const __nv_bfloat16*)dO, idx, sink, scale,           \
                                        (const __nv_bfloat16*)o, lse, dq, dkv, dsink, sq, H,  \
                                        n_c, ratio, window, K, status, doc, tb, te, njobs);   \
    count_launches(1);                                                                        \
  }
  if (QB == 8) CSA_TC_BWD(8)
  else if (QB == 4) CSA_TC_BWD(4)
  else CSA_TC_BWD(2)
#undef CSA_TC_BWD
  return cudaGetLastError();
}

}  // namespace csa
