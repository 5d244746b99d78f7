// Sparse MQA forward on the 5th-generation tensor cores (tcgen05 + TMEM) at
// the production width: bf16, d = 512, H = 64.
//
// Semantics as csa_attn_fwd ("Add unfused SBHD compressed sparse attention":
// unfused sparse core, sink parameter; "Refactor Deepseek v4 to use Attention
// Gym's Compressed Sparse Attention": window + selected entries + sink in one
// softmax, per-head LSE; its DeepSeek-V4 shape: 64 heads of width 512).
//
// At d = 512 the output of 128 (query, head) rows would fill all 512 TMEM
// columns, so the products are formed transposed, one query per CTA:
//   S^T [slots, heads] = KV [slots, d] . Q^T         (M = 128 slots, N = 64, K = 512)
//   O^T [d, heads]    += KV^T [d, slots] . P^T       (four M = 128 tiles of d, N = 64)
// S^T takes 64 TMEM columns and O^T 256.  The KV tile (128 gathered rows x
// 512, 128 KB, 128-byte-swizzled K-major) is the K-major A operand of S^T
// and, read MN-major, the A operand of O^T; Q (64 KB, by TMA) is the K-major
// B operand of S^T; P (16 KB, one 128-byte row of 64 heads per slot) is the
// MN-major B operand of O^T.
//
// Each thread owns one slot (TMEM lane) and 16 heads in the softmax, so the
// per-head maximum and sum over a tile's 128 slots are reductions across
// lanes: a transposing butterfly (16 shuffles) leaves lanes l and l + 16 with
// head l's value, and four shared-memory entries per head join the lane
// quarters.  O is normalized by the sum of the bf16-rounded probabilities
// that enter its product (a convex combination), the LSE by the exact sum.
// The running maximum is kept per head; O^T and the sums are rescaled only
// when a head's maximum grows by more than 2^8 (the sink is the initial
// state: m = sink, mass 1).  Slots are the query's window rows followed by
// its valid selected entries (a repeated entry is a repeated slot).
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"

#include <cudaTypedefs.h>

namespace csa {
namespace atd {

using namespace csa::umma;

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kSlots = 128;
constexpr int kThreads = 512;                  // 16 warps: TMEM lane quarter x head quarter
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 128;     // S^T: 64 columns; O^T: 4 x 64 columns
constexpr uint32_t kQBlk = kH * 128;           // 8 KB: 64 head rows of 128 B
constexpr uint32_t kKvBlk = kSlots * 128;      // 16 KB: 128 slot rows of 128 B
constexpr float kRescale = 8.f;                // lazy rescale threshold (log2 domain)
constexpr int kGather = kThreads - 32;         // warps 1-15 gather the KV tiles

struct Layout {
  static constexpr uint32_t Q = 0;                       // [8][64 rows][128 B]
  static constexpr uint32_t KV = 8 * kQBlk;              // [8][128 rows][128 B]
  static constexpr uint32_t P = KV + 8 * kKvBlk;         // [128 rows][128 B]
  static constexpr uint32_t BARS = P + kSlots * 128;     // q, s, kv[4], o[4]
  static constexpr uint32_t TSLOT = BARS + 10 * 8;
  static constexpr uint32_t FLAG = TSLOT + 8;            // any-rescale flag, slot count
  static constexpr uint32_t RED = FLAG + 8;              // [2][4][64] floats
  static constexpr uint32_t MRUN = RED + 8 * kH * 4;     // [64] running max (log2)
  static constexpr uint32_t FAC = MRUN + kH * 4;         // [64] rescale factor of the tile
  static constexpr uint32_t LSINK = FAC + kH * 4;        // [64] sink mass
  static constexpr uint32_t ROWS = LSINK + kH * 4;       // slot rows
};

// Swizzled offset of 16-byte chunk ch (0..63) of 512-element row r of the
// KV tile (eight 64-element K blocks of 128 rows).
__device__ __forceinline__ uint32_t kv_off(int r, int ch) {
  return (uint32_t)((ch >> 3) * kKvBlk + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// 16-byte asynchronous copy that reads src_bytes (16 or 0) and zero-fills
// the rest: a padding slot becomes zeros through the same copy path.
__device__ __forceinline__ void cp_async_16_zfill(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Transposing butterfly over the 32 lanes: v[c] (c < 16) holds this lane's
// value of column c; afterwards lanes l and l + 16 hold op over all 32 lanes
// of column l % 16.
template <bool kMax>
__device__ __forceinline__ float lane_transpose_reduce16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 8, n = 8; off >= 1; off >>= 1, n >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = up ? v[i] : v[i + n];
      const float keep = up ? v[i + n] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  const float other = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return kMax ? fmaxf(v[0], other) : v[0] + other;
}

__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc512_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __nv_bfloat16* __restrict__ kv,
    const int32_t* __restrict__ idx, const float* __restrict__ sink, float scale,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int sq, int n_c, int ratio,
    int window, int K, int* __restrict__ status, const int32_t* __restrict__ doc, int tb,
    int te) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + Layout::BARS);
  uint64_t* bar_s = bar_q + 1;          // S^T of the tile complete
  uint64_t* bar_kv = bar_q + 2;         // [4] the tile's d-block pair mt gathered
  uint64_t* bar_of = bar_q + 6;         // [4] O^T M-tile mt of the tile complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::TSLOT);
  int* flag = reinterpret_cast<int*>(sm + Layout::FLAG);
  float* red = reinterpret_cast<float*>(sm + Layout::RED);
  float* m_run = reinterpret_cast<float*>(sm + Layout::MRUN);
  float* fac = reinterpret_cast<float*>(sm + Layout::FAC);
  float* lsink = reinterpret_cast<float*>(sm + Layout::LSINK);
  int* rows = reinterpret_cast<int*>(sm + Layout::ROWS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = (int)gridDim.x / (te - tb);
  const int bi = (int)blockIdx.x % b;
  const int t = te - 1 - (int)blockIdx.x / b;           // heaviest queries first
  const int n_kv = sq + n_c;
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * kD;

  // ---- set-up: barriers, TMEM, Q tile (TMA), slot list, softmax state ------
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_s, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bar_kv[i], kGather);
      mbar_init(&bar_of[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  if (tid < kH) {
    const bool has_sink = sink != nullptr;
    m_run[tid] = has_sink ? sink[tid] * kLog2e : -INFINITY;
    lsink[tid] = has_sink ? 1.f : 0.f;
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    mbar_expect_tx(bar_q, 8 * kQBlk);
    const int row0 = (bi * sq + t) * kH;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) tma_load_2d(sm + Layout::Q + kb * kQBlk, &tmap_q, bar_q,
                                               kb * 64, row0);
  }
  if (warp == 0) {
    const int c = build_slots_warp(rows, idx ? idx + ((long long)bi * sq + t) * K : nullptr, K, t,
                                   sq, n_c, ratio, window, doc ? doc + (long long)bi * sq : nullptr);
    if (lane == 0) flag[1] = c;
  }
  __syncthreads();
  const int S_total = flag[1];
  const int ntiles = (S_total + kSlots - 1) / kSlots;

  const int qd = warp & 3, hq = warp >> 2;             // lane quarter, head quarter
  const int r = qd * 32 + lane;                        // TMEM lane: slot (S^T) or d (O^T)
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const float sc2 = scale * kLog2e;
  float l_part[16], lr_part[16];                       // this slot lane's mass per head:
#pragma unroll                                         // exact, and of the rounded P
  for (int c = 0; c < 16; ++c) l_part[c] = lr_part[c] = 0.f;

  bool ok = __syncthreads_and(mbar_wait(bar_q, 0));
  int site = ok ? 0 : kSiteFwdQ;
  bool fail = false;                                   // a bounded wait of this thread gave up

  // Gather of tile it by warps 1-15, one pair of 64-wide d blocks at a time:
  // pair mt of the KV buffer is free once the previous tile's O^T M-tile mt
  // (which reads those blocks) has completed; its arrival is signalled on
  // bar_kv[mt] so that the S^T K-steps over it can start.  Padding slots past
  // the list are zero-filled by the same copies.
  auto gather = [&](int it) {
    const int g = tid - 32;
    const int sbase = it * kSlots;
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      bool good = true;
      if (it > 0) good = mbar_wait(&bar_of[mt], (it - 1) & 1);
      fail |= !good;
      if (good) {
        for (int c = g; c < kSlots * 16; c += kGather) {
          const int rr = c >> 4, ch = mt * 16 + (c & 15);
          const int s = sbase + rr;
          const bool pad = s >= S_total;
          const __nv_bfloat16* src = kv_b + (pad ? 0ll : (long long)rows[s] * kD) + ch * 8;
          cp_async_16_zfill(sm + Layout::KV + kv_off(rr, ch), src, pad ? 0u : 16u);
        }
      }
      cp_async_commit();
      if (mt > 0) {
        cp_async_wait_group<1>();
        fence_proxy_async_smem();
        mbar_arrive(&bar_kv[mt - 1]);
      }
    }
    cp_async_wait_group<0>();
    fence_proxy_async_smem();
    mbar_arrive(&bar_kv[3]);
  };
  // S^T of tile it, issued by one thread pair by pair as the gather lands
  auto issue_s = [&](int it) {
    constexpr uint32_t idesc = idesc_bf16_f32_major(kSlots, kH, 0, 0);
    const uint32_t kva = smem_addr(sm + Layout::KV), qa = smem_addr(sm + Layout::Q);
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      if (!mbar_wait(&bar_kv[mt], it & 1)) {
        fail = true;
        return;
      }
      fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int k = mt * 8 + kk;
        const uint32_t ka = kva + (k >> 2) * kKvBlk + (k & 3) * 32;
        const uint32_t qb = qa + (k >> 2) * kQBlk + (k & 3) * 32;
        mma_bf16_ss(tmem + kColS, sw128_desc(ka), sw128_desc(qb), idesc, k > 0 ? 1u : 0u);
      }
    }
    mma_commit(bar_s);
  };
  if (ok && ntiles > 0) {
    if (warp > 0) gather(0);
    else if (lane == 0) issue_s(0);
  }

  for (int it = 0; it < ntiles && ok; ++it) {
    __syncwarp();
    ok = __syncthreads_and(mbar_wait(bar_s, it & 1) && !fail);
    if (!ok) { site = kSiteFwdS; break; }
    fence_after();
    const int sbase = it * kSlots;

    // ---- softmax over the tile's slots, per head --------------------------
    const float bias = sbase + r < S_total ? 0.f : -INFINITY;
    float x[16];
    {
      uint32_t v[16];
      tmem_ld16_wait(tmem + lane_base + kColS + hq * 16, v);
#pragma unroll
      for (int c = 0; c < 16; ++c) x[c] = fmaf(__uint_as_float(v[c]), sc2, bias);
    }
    {
      float mx[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) mx[c] = x[c];
      const float m = lane_transpose_reduce16<true>(mx);
      if (lane < 16) red[qd * kH + hq * 16 + lane] = m;
    }
    if (tid == 0) flag[0] = 0;
    __syncthreads();
    if (tid < kH) {
      const float mt = fmaxf(fmaxf(red[tid], red[kH + tid]),
                             fmaxf(red[2 * kH + tid], red[3 * kH + tid]));
      const float mo = m_run[tid];
      float f = 1.f;
      if (mt > mo + kRescale || (mo == -INFINITY && mt != -INFINITY)) {
        f = ex2(mo - mt);                              // 0 when mo = -inf
        m_run[tid] = mt;
        lsink[tid] *= f;
        flag[0] = 1;
      }
      fac[tid] = f;
    }
    __syncthreads();
    if (flag[0]) {                                     // CTA-uniform
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        l_part[c] *= fac[hq * 16 + c];
        lr_part[c] *= fac[hq * 16 + c];
      }
      if (it > 0) {
        // rescale O^T: this thread's d lane of M-tile hq, all heads (the
        // previous tile's MMAs into it have completed; the wait returns at once)
        if (!mbar_wait(&bar_of[hq], (it - 1) & 1)) fail = true;
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t ta = tmem + lane_base + kColO + hq * kH + h2 * 32;
          uint32_t v[32];
          tmem_ld32_wait(ta, v);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            v[c] = __float_as_uint(__uint_as_float(v[c]) * fac[h2 * 32 + c]);
          CSA_TMEM_ST32(ta, v);
          tmem_wait_st();
        }
      }
    }
    // P = 2^(x - m) as bf16 into this slot's row of the P tile (this thread's
    // 16 heads: 32 bytes = 2 swizzled 16-byte chunks)
    unsigned char* prow = sm + Layout::P + r * 128;
#pragma unroll
    for (int c8 = 0; c8 < 2; ++c8) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int c = c8 * 8 + e;
        const float p0 = ex2(x[c] - m_run[hq * 16 + c]);   // masked slots: 2^-inf = 0
        const float p1 = ex2(x[c + 1] - m_run[hq * 16 + c + 1]);
        l_part[c] += p0;
        l_part[c + 1] += p1;
        const __nv_bfloat162 h2v = __floats2bfloat162_rn(p0, p1);
        const float2 back = __bfloat1622float2(h2v);
        lr_part[c] += back.x;
        lr_part[c + 1] += back.y;
        pk[e / 2] = *reinterpret_cast<const uint32_t*>(&h2v);
      }
      *reinterpret_cast<uint4*>(prow + ((((hq * 2 + c8) ^ (r & 7))) << 4)) =
          make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0) {
      fence_after();
      // O^T[d, h] += KV^T[d, slots] P^T[slots, h]: A = KV read MN-major (the
      // two 64-wide d blocks of M-tile mt, 16 slot rows per K step), B = P
      // read MN-major (one 64-head atom per slot row)
      constexpr uint32_t idesc = idesc_bf16_f32_major(kD / 4, kH, 1, 1);
      const uint32_t kva = smem_addr(sm + Layout::KV), pa = smem_addr(sm + Layout::P);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int k = 0; k < kSlots / 16; ++k) {
          const uint64_t a = sw128_desc_mn(kva + 2 * mt * kKvBlk + k * 2048, kKvBlk);
          const uint64_t bdesc = sw128_desc_mn(pa + k * 2048, kKvBlk);
          mma_bf16_ss(tmem + kColO + mt * kH, a, bdesc, idesc, (it > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&bar_of[mt]);
      }
    }
    // the next tile's gather streams in behind these MMAs, and its S^T
    // follows the gather
    if (it + 1 < ntiles) {
      if (warp > 0) gather(it + 1);
      else if (lane == 0) issue_s(it + 1);
    }
  }
  __syncwarp();
  if (ok && ntiles > 0) {
    ok = __syncthreads_and(mbar_wait(&bar_of[hq], (ntiles - 1) & 1) && !fail);
    if (!ok) site = kSiteFwdLast;
  }
  cp_async_wait_all_();                                // no copy in flight past this point
  if (!ok && tid == 0) set_status(status, kDevTimeout, site);
  fence_after();

  // ---- epilogue: per-head mass, LSE, O = O^T^T / l ------------------------------
  {
    const float le = lane_transpose_reduce16<false>(l_part);
    const float lr = lane_transpose_reduce16<false>(lr_part);
    if (lane < 16) {
      red[qd * kH + hq * 16 + lane] = le;
      red[4 * kH + qd * kH + hq * 16 + lane] = lr;
    }
  }
  __syncthreads();
  if (tid < kH) {
    const float l_tot = (red[tid] + red[kH + tid]) + (red[2 * kH + tid] + red[3 * kH + tid]) +
                        lsink[tid];
    const float* rr = red + 4 * kH;
    const float lr_tot = (rr[tid] + rr[kH + tid]) + (rr[2 * kH + tid] + rr[3 * kH + tid]) +
                         lsink[tid];
    fac[tid] = 1.f / lr_tot;
    if (ok) lse[((long long)bi * sq + t) * kH + tid] = (m_run[tid] + log2f(l_tot)) * kLn2;
  }
  __syncthreads();
  if (ok) {
    __nv_bfloat16* orow = o + ((long long)bi * sq + t) * kH * kD;
    const int dcol = hq * 128 + r;                     // this thread's d
#pragma unroll 1
    for (int h4 = 0; h4 < 4; ++h4) {
      uint32_t v[16];
      tmem_ld16_wait(tmem + lane_base + kColO + hq * kH + h4 * 16, v);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int h = h4 * 16 + c;
        orow[(long long)h * kD + dcol] = __float2bfloat16_rn(__uint_as_float(v[c]) * fac[h]);
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace atd

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_512() {
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

size_t attn_tc512_smem(int window, int Kl) {
  return 1024 + atd::Layout::ROWS + (size_t)(window + Kl + 32) * sizeof(int);
}
}  // namespace

// The production-width tensor-core forward applies to bf16, d = 512, H = 64,
// with the slot list (window + K entries) within shared memory.
bool attn_tc512_supported(int H, int d, int window, int Kl) {
  if (d != atd::kD || H != atd::kH) return false;
  if (encode_fn_512() == nullptr) return false;
  return attn_tc512_smem(window, Kl) <= 227 * 1024;
}

cudaError_t launch_attn_fwd_tc512(const void* q, const void* kv, const int32_t* idx,
                                  const float* sink, float scale, void* o, float* lse, int b,
                                  int sq, int n_c, int ratio, int window, int K, int* status,
                                  cudaStream_t s, const int32_t* doc, int tb, int te) {
  auto encode = encode_fn_512();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tq;
  const cuuint64_t dims[2] = {(cuuint64_t)atd::kD, (cuuint64_t)b * sq * atd::kH};
  const cuuint64_t strides[1] = {(cuuint64_t)atd::kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)atd::kH};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int Kl = idx ? K : n_c;
  const size_t smem = attn_tc512_smem(window, Kl);
  auto k = atd::attn_fwd_tc512_kernel;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k<<<(unsigned)((te - tb) * b), atd::kThreads, smem, s>>>(
      tq, (const __nv_bfloat16*)kv, idx, sink, scale, (__nv_bfloat16*)o, lse, sq, n_c, ratio,
      window, K, status, doc, tb, te);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
