// Sparse MQA backward on the 5th-generation tensor cores (tcgen05 + TMEM) at
// the production width: bf16, d = 512, H = 64.
//
// Semantics as csa_attn_bwd ("Add unfused SBHD compressed sparse attention",
// review of the gather backward: compact [b*n_kv, d] dKV with repeated
// indices summed; "Add the min-memory DSA attention kernels": fp32 scatter):
//   D = sum_i p_i dP_i,  p_i = exp(s_i - lse),  ds_i = p_i (dP_i - D),
//   dq = scale sum_i ds_i kv_i,  dkv_i += p_i dO + scale ds_i q,
//   dsink = -exp(sink - lse) D.
//
// One query per CTA, products transposed as in the production-width forward
// (slots on TMEM lanes, the query's 64 heads on columns):
//   S^T = KV Q^T, dP^T = KV dO^T          (M = 128 slots, N = 64, K = 512)
//   dQ^T [d, h] += KV^T dS^T              (four M = 128 tiles of d)
//   dKV [slots, d] = P^T dO + dS^T Q      (M = 128 slots, N = 128 d at a time)
// TMEM: S^T 64 columns, dP^T 64, dQ^T 256, one 128-column dKV chunk; the
// chunks of odd pairs use those 128 columns and the chunks of even pairs the
// S^T / dP^T columns (free once P and dS are formed), so that a chunk is
// drained into the compact buffer while the next pair's MMAs run.
// Q, dO and the tile's KV rows do not fit shared memory together with P and
// dS (320 KB), so all three stream through it in pairs of 64-wide d blocks
// (128 d: the KV rows of the tile 32 KB, Q and dO 16 KB each, the last two
// by TMA from L2): the S^T / dP^T K-steps and the dQ^T M-tile / dKV chunk of
// a pair run on the pair in place.  Two 64 KB stages: the next pair streams
// in while the tensor core works on the current one.  Pass 1 forms D = sum p dP exactly; pass 2
// forms P and dS * scale as bf16 hi + lo (about 16 significant bits, so the
// fp32 sums of hot rows over thousands of queries stay accurate), then per
// pair dQ^T and the tile's dKV chunk, which is added into the compact buffer
// with fp32 vector reductions.
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"

#include <cudaTypedefs.h>

namespace csa {
namespace atdb {

using namespace csa::umma;

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kSlots = 128;
constexpr int kThreads = 512;                   // 16 warps: TMEM lane quarter x head quarter
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kColDKV = 384;
__device__ __forceinline__ uint32_t dkv_col(int p) { return (p & 1) ? kColDKV : kColS; }
constexpr uint32_t kKvBlk = kSlots * 128;       // 16 KB: 128 slot rows of 128 B
constexpr uint32_t kHBlk = kH * 128;            // 8 KB: 64 head rows of 128 B

constexpr uint32_t kStage = 2 * kKvBlk + 4 * kHBlk;   // 64 KB: KV, Q, dO of one d pair

struct Layout {
  // stage st at st * kStage: KV pair [2][128 rows][128 B], then Q pair
  // [2][64 rows][128 B], then dO pair
  static constexpr uint32_t KV = 0;
  static constexpr uint32_t Q = 2 * kKvBlk;              // within a stage
  static constexpr uint32_t G = Q + 2 * kHBlk;           // within a stage
  static constexpr uint32_t PH = 2 * kStage;             // [128 slot rows][128 B]
  static constexpr uint32_t PL = PH + kKvBlk;
  static constexpr uint32_t DH = PL + kKvBlk;
  static constexpr uint32_t DL = DH + kKvBlk;
  static constexpr uint32_t BARS = DL + kKvBlk;          // ld[2], mma
  static constexpr uint32_t TSLOT = BARS + 3 * 8;
  static constexpr uint32_t SCAL = TSLOT + 8;            // slot count
  static constexpr uint32_t RED = SCAL + 8;              // [4][64] floats
  static constexpr uint32_t LSE2 = RED + 4 * kH * 4;     // [64]
  static constexpr uint32_t DROW = LSE2 + kH * 4;        // [64]
  static constexpr uint32_t ROWS = DROW + kH * 4;        // slot rows
};

__device__ __forceinline__ void cp_async_16_zfill(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// Transposing butterfly (as in the forward): v[c] (c < 16) of every lane ->
// lanes l and l + 16 hold the sum over the 32 lanes of column l % 16.
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

// Store 8 values as bf16 hi and bf16 residual at byte offset off of X and Y.
__device__ __forceinline__ void store_hi_lo8(unsigned char* X, unsigned char* Y, uint32_t off,
                                             const float* v) {
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

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_tc512_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_do,
    const __nv_bfloat16* __restrict__ kv, const int32_t* __restrict__ idx,
    const float* __restrict__ sink, float scale, const float* __restrict__ lse,
    float* __restrict__ dq, float* __restrict__ dkv, float* __restrict__ dsink, int sq, int n_c,
    int ratio, int window, int K, int* __restrict__ status, const int32_t* __restrict__ doc,
    int tb, int te) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + Layout::BARS);   // [2] Q / dO by TMA
  uint64_t* bar_mma = bar_ld + 2;                                       // MMA group done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::TSLOT);
  int* scal = reinterpret_cast<int*>(sm + Layout::SCAL);
  float* red = reinterpret_cast<float*>(sm + Layout::RED);
  float* lse2_s = reinterpret_cast<float*>(sm + Layout::LSE2);
  float* D_s = reinterpret_cast<float*>(sm + Layout::DROW);
  int* rows = reinterpret_cast<int*>(sm + Layout::ROWS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = (int)gridDim.x / (te - tb);
  const int bi = (int)blockIdx.x % b;
  const int t = te - 1 - (int)blockIdx.x / b;           // heaviest queries first
  const int n_kv = sq + n_c;
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * kD;
  float* dkv_b = dkv + (long long)bi * n_kv * kD;
  const long long qrow = ((long long)bi * sq + t) * kH;

  if (tid == 0) {
    mbar_init(&bar_ld[0], 1);
    mbar_init(&bar_ld[1], 1);
    mbar_init(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid < kH) lse2_s[tid] = lse[qrow + tid] * kLog2e;
  if (warp == 1) {
    const int c = build_slots_warp(rows, idx ? idx + ((long long)bi * sq + t) * K : nullptr, K, t,
                                   sq, n_c, ratio, window, doc ? doc + (long long)bi * sq : nullptr);
    if (lane == 0) scal[0] = c;
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const int S_total = scal[0];
  const int ntiles = (S_total + kSlots - 1) / kSlots;

  const int qd = warp & 3, hq = warp >> 2;             // lane quarter, head quarter
  const int r = qd * 32 + lane;                        // TMEM lane: slot or d
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const float sc2 = scale * kLog2e;
  uint32_t n_mma = 0;                                  // completed phases of bar_mma
  int n_issued = 0, n_waited = 0;                      // jobs whose stage was issued / waited
  bool ok = true;
  int site = 0;

  // The jobs of the query, in order: pass 1 (D) runs S^T / dP^T over the four
  // d pairs of every tile; pass 2 runs, per tile, S^T / dP^T over the pairs,
  // then dQ^T / dKV over the pairs.  Job j streams its pair into stage j & 1.
  const int J1 = 4 * ntiles, J = 12 * ntiles;
  auto job = [&](int j, int* it, int* p, bool* sdp) {
    if (j < J1) {
      *it = j >> 2; *p = j & 3; *sdp = true;
    } else {
      const int jj = j - J1;
      *it = jj >> 3; *p = jj & 3; *sdp = (jj & 7) < 4;
    }
  };
  // Issue the copies of job j's pair into stage j & 1: the tile's KV rows
  // (every thread, 16-byte copies, padding slots zero-filled) and the
  // query's Q and dO (thread 0, TMA).
  auto stage_issue = [&](int j) {
    int it, p;
    bool sdp;
    job(j, &it, &p, &sdp);
    unsigned char* st = sm + (j & 1) * kStage;
    const int sbase = it * kSlots;
    ++n_issued;
    for (int c = tid; c < kSlots * 16; c += kThreads) {
      const int rr = c >> 4, chp = c & 15;              // chunk within the pair's 128 d
      const int s = sbase + rr;
      const bool pad = s >= S_total;
      const __nv_bfloat16* src = kv_b + (pad ? 0ll : (long long)rows[s] * kD) + p * 128 + chp * 8;
      const uint32_t off = (chp >> 3) * kKvBlk + rr * 128 + ((((chp & 7) ^ (rr & 7))) << 4);
      cp_async_16_zfill(st + Layout::KV + off, src, pad ? 0u : 16u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (tid == 0) {
      uint64_t* bl = &bar_ld[j & 1];
      mbar_expect_tx(bl, 4 * kHBlk);
      tma_load_2d(st + Layout::Q, &tmap_q, bl, p * 128, (int)qrow);
      tma_load_2d(st + Layout::Q + kHBlk, &tmap_q, bl, p * 128 + 64, (int)qrow);
      tma_load_2d(st + Layout::G, &tmap_do, bl, p * 128, (int)qrow);
      tma_load_2d(st + Layout::G + kHBlk, &tmap_do, bl, p * 128 + 64, (int)qrow);
    }
  };
  // Wait for job j's stage (its copies are the only ones in flight here).
  auto stage_wait = [&](int j) -> bool {
    cp_async_wait_all_();
    fence_proxy_async_smem();
    const bool got = mbar_wait(&bar_ld[j & 1], (j >> 1) & 1);
    ++n_waited;
    fence_before();
    return __syncthreads_and(got);
  };

  // add a slot's 128 d of a pair's dKV chunk into its compact dKV row
  // (warp (qd, hq) takes 32 of the columns)
  auto drain = [&](int it, int p) {
    uint32_t v[32];
    tmem_ld32_wait(tmem + lane_base + dkv_col(p) + hq * 32, v);
    const int s = it * kSlots + r;
    if (s < S_total) {
      float* dst = dkv_b + (long long)rows[s] * kD + p * 128 + hq * 32;
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        red_add_v4(dst + c, __uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                   __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
    }
  };
  int def_it = -1, def_p = 0;                          // the chunk waiting to be drained

  float dpart[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) dpart[c] = 0.f;
  float Dh[16];
  if (J > 0) stage_issue(0);
  for (int j = 0; j < J && ok; ++j) {
    int it, p;
    bool sdp;
    job(j, &it, &p, &sdp);
    if (!stage_wait(j)) { ok = false; site = kSiteBwdQ; break; }
    if (tid == 0) {
      fence_after();
      const uint32_t st = smem_addr(sm + (j & 1) * kStage);
      const uint32_t kva = st + Layout::KV, qa = st + Layout::Q, ga = st + Layout::G;
      if (sdp) {
        // S^T += KV_p Q_p^T and dP^T += KV_p dO_p^T over the pair's 128 d
        constexpr uint32_t idesc = idesc_bf16_f32_major(kSlots, kH, 0, 0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t ka = kva + (k >> 2) * kKvBlk + (k & 3) * 32;
          const uint32_t qo = (k >> 2) * kHBlk + (k & 3) * 32;
          const uint32_t acc = (p > 0 || k > 0) ? 1u : 0u;
          mma_bf16_ss(tmem + kColS, sw128_desc(ka), sw128_desc(qa + qo), idesc, acc);
          mma_bf16_ss(tmem + kColDP, sw128_desc(ka), sw128_desc(ga + qo), idesc, acc);
        }
      } else {
        const uint32_t pha = smem_addr(sm + Layout::PH), pla = smem_addr(sm + Layout::PL);
        const uint32_t dha = smem_addr(sm + Layout::DH), dla = smem_addr(sm + Layout::DL);
        // dQ^T[d, h] += KV^T[d, slots] dS^T[slots, h]: A = the KV pair read
        // MN-major (its two 64-wide d blocks), B = dS read MN-major
        constexpr uint32_t idesc_q = idesc_bf16_f32_major(kSlots, kH, 1, 1);
#pragma unroll
        for (int k = 0; k < kSlots / 16; ++k) {
          const uint64_t a = sw128_desc_mn(kva + k * 2048, kKvBlk);
          mma_bf16_ss(tmem + kColDQ + p * kH, a, sw128_desc_mn(dha + k * 2048, kKvBlk), idesc_q,
                      (it > 0 || k > 0) ? 1u : 0u);
          mma_bf16_ss(tmem + kColDQ + p * kH, a, sw128_desc_mn(dla + k * 2048, kKvBlk), idesc_q,
                      1u);
        }
        // dKV[slots, d] = P^T dO + dS^T Q over the heads: A = P / dS rows
        // (K-major, heads contiguous), B = dO / Q pair read MN-major
        constexpr uint32_t idesc_kv = idesc_bf16_f32_major(kSlots, 128, 0, 1);
#pragma unroll
        for (int k = 0; k < kH / 16; ++k) {
          const uint64_t bg = sw128_desc_mn(ga + k * 2048, kHBlk);
          const uint64_t bq = sw128_desc_mn(qa + k * 2048, kHBlk);
          const uint32_t dc = tmem + dkv_col(p);
          mma_bf16_ss(dc, sw128_desc(pha + k * 32), bg, idesc_kv, k > 0 ? 1u : 0u);
          mma_bf16_ss(dc, sw128_desc(pla + k * 32), bg, idesc_kv, 1u);
          mma_bf16_ss(dc, sw128_desc(dha + k * 32), bq, idesc_kv, 1u);
          mma_bf16_ss(dc, sw128_desc(dla + k * 32), bq, idesc_kv, 1u);
        }
      }
      mma_commit(bar_mma);
    }
    // the next job's pair streams into the other stage (the MMAs that read it
    // last, those of job j - 1, have completed), and the previous chunk is
    // drained while these MMAs run
    if (j + 1 < J) stage_issue(j + 1);
    if (def_it >= 0) {
      drain(def_it, def_p);
      def_it = -1;
    }
    ok = __syncthreads_and(mbar_wait(bar_mma, n_mma & 1));
    ++n_mma;
    if (!ok) { site = sdp ? kSiteBwdS : kSiteBwdDS; break; }
    fence_after();

    if (sdp && p == 3) {
      const float bias = it * kSlots + r < S_total ? 0.f : -INFINITY;
      uint32_t vs[16], vp[16];
      tmem_ld16_wait(tmem + lane_base + kColS + hq * 16, vs);
      tmem_ld16_wait(tmem + lane_base + kColDP + hq * 16, vp);
      if (j < J1) {
        // pass 1: D = sum p dP
#pragma unroll
        for (int c = 0; c < 16; ++c)
          dpart[c] = fmaf(ex2(fmaf(__uint_as_float(vs[c]), sc2, bias - lse2_s[hq * 16 + c])),
                          __uint_as_float(vp[c]), dpart[c]);
      } else {
        // pass 2: P and dS * scale (hi + lo) into this slot's rows of PH/PL, DH/DL
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          float pv[8], dv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = c8 * 8 + e;
            pv[e] = ex2(fmaf(__uint_as_float(vs[c]), sc2, bias - lse2_s[hq * 16 + c]));
            dv[e] = pv[e] * (__uint_as_float(vp[c]) - Dh[c]) * scale;
          }
          const uint32_t off = r * 128 + ((((hq * 2 + c8) ^ (r & 7))) << 4);
          store_hi_lo8(sm + Layout::PH, sm + Layout::PL, off, pv);
          store_hi_lo8(sm + Layout::DH, sm + Layout::DL, off, dv);
        }
        fence_proxy_async_smem();
      }
      fence_before();
      __syncthreads();                                 // S^T / dP^T read before they are rewritten
      if (j == J1 - 1) {
        // end of pass 1: D per head
        const float v = lane_transpose_sum16(dpart);
        if (lane < 16) red[qd * kH + hq * 16 + lane] = v;
        __syncthreads();
        if (tid < kH)
          D_s[tid] = (red[tid] + red[kH + tid]) + (red[2 * kH + tid] + red[3 * kH + tid]);
        __syncthreads();
#pragma unroll
        for (int c = 0; c < 16; ++c) Dh[c] = D_s[hq * 16 + c];
      }
    } else if (!sdp) {
      // drained during the next job (the chunk's columns are next written
      // two jobs later, after at least one more barrier)
      def_it = it;
      def_p = p;
    }
  }
  if (ok && def_it >= 0) drain(def_it, def_p);
  cp_async_wait_all_();                                // no copy in flight past this point
  for (int j = n_waited; !ok && j < n_issued; ++j)     // nor a TMA load (bounded waits)
    mbar_wait(&bar_ld[j & 1], (j >> 1) & 1);
  if (!ok && tid == 0) set_status(status, kDevTimeout, site);

  // ---- dq rows and the sink gradient --------------------------------------------
  if (ok && ntiles > 0) {
    float* dqrow = dq + qrow * kD;
    const int dcol = hq * 128 + r;
#pragma unroll 1
    for (int h4 = 0; h4 < 4; ++h4) {
      uint32_t v[16];
      tmem_ld16_wait(tmem + lane_base + kColDQ + hq * kH + h4 * 16, v);
#pragma unroll
      for (int c = 0; c < 16; ++c) dqrow[(long long)(h4 * 16 + c) * kD + dcol] = __uint_as_float(v[c]);
    }
    if (sink != nullptr && tid < kH)
      atomicAdd(&dsink[tid], -exp2f(sink[tid] * kLog2e - lse2_s[tid]) * D_s[tid]);
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace atdb

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_512b() {
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

size_t attn_tc512_bwd_smem(int window, int Kl) {
  return 1024 + atdb::Layout::ROWS + (size_t)(window + Kl + 32) * sizeof(int);
}

bool make_map_512(CUtensorMap* m, const void* base, long long rows) {
  auto encode = encode_fn_512b();
  if (encode == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)atdb::kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)atdb::kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)atdb::kH};
  const cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}
}  // namespace

// The production-width tensor-core backward applies to bf16, d = 512, H = 64
// with the slot list within shared memory.
bool attn_tc512_bwd_supported(int H, int d, int window, int Kl) {
  if (d != atdb::kD || H != atdb::kH) return false;
  if (encode_fn_512b() == nullptr) return false;
  return attn_tc512_bwd_smem(window, Kl) <= 227 * 1024;
}

cudaError_t launch_attn_bwd_tc512(const void* q, const void* kv, const int32_t* idx,
                                  const float* sink, float scale, const float* lse,
                                  const void* dO, float* dq, float* dkv, float* dsink, int b,
                                  int sq, int n_c, int ratio, int window, int K, int* status,
                                  cudaStream_t s, const int32_t* doc, int tb, int te) {
  CUtensorMap tq, tg;
  const long long rows = (long long)b * sq * atdb::kH;
  if (!make_map_512(&tq, q, rows) || !make_map_512(&tg, dO, rows)) return cudaErrorInvalidValue;
  const int Kl = idx ? K : n_c;
  const size_t smem = attn_tc512_bwd_smem(window, Kl);
  auto k = atdb::attn_bwd_tc512_kernel;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k<<<(unsigned)((te - tb) * b), atdb::kThreads, smem, s>>>(
      tq, tg, (const __nv_bfloat16*)kv, idx, sink, scale, lse, dq, dkv, dsink, sq, n_c, ratio,
      window, K, status, doc, tb, te);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
