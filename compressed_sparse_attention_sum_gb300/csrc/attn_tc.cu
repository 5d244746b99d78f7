// Sparse MQA forward on the 5th-generation tensor cores (tcgen05 + TMEM),
// bf16, d = 128.
//
// Semantics as csa_attn_fwd ("Add unfused SBHD compressed sparse attention":
// unfused sparse core, sink parameter; "Refactor Deepseek v4 to use Attention
// Gym's Compressed Sparse Attention": window + selected entries + sink in one
// softmax, per-head LSE).
//
// One CTA owns 128 rows = QB consecutive queries x H heads (H * QB = 128), so
// the rows of the score tile are (query, head) pairs and each thread owns one
// row (one TMEM lane): the softmax needs no cross-thread reduction.  The CTA
// walks the union of its queries' slots: the window rows of the block (one
// contiguous run of raw rows) and the sorted union of the blocks the queries
// selected.  Each query sees the union through a per-query multiplicity
// count: 0 masks the slot, c >= 1 adds log2(c) to the logit (a block listed
// twice is two softmax terms).  Selections of neighbouring queries overlap
// heavily, so one gathered KV tile serves all QB queries.
//
// Per tile of 128 slots: 16-byte cp.async gather of the KV rows into the
// 128-byte-swizzled K-major layout; one thread issues S = Q K^T (M=128 rows,
// N=128 slots, K=128) into TMEM; every thread reads its row of S, applies
// scale, mask and bias, updates its running max (rescaling O only when the
// max grows by more than 2^8, else keeping the stale max), writes P (bf16)
// to shared memory; one thread issues O += P V with the same KV tile as the
// MN-major B operand (N = d, K = slots).  The sink is the initial running
// state (m = sink, l = 1): it enters the denominator only.
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"
#include "attn_union.cuh"

#include <cudaTypedefs.h>

namespace csa {
namespace atc {

using namespace csa::umma;

constexpr int kRows = 128;
constexpr int kSlots = 128;
constexpr int kD = 128;
constexpr int kThreads = 256;                   // 8 warps: TMEM lane quarter x column half
constexpr uint32_t kTmemCols = 256;            // S: columns 0..127, O: 128..255
constexpr uint32_t kBlk = kRows * 128;          // one 64-wide K block of a 128-row tile (16 KB)
constexpr float kRescale = 8.f;                 // lazy rescale threshold (log2 domain)

struct Layout {
  // byte offsets from the 1024-aligned base
  static constexpr uint32_t Q = 0;              // [2][128 rows][128 B]
  static constexpr uint32_t KV = 2 * kBlk;      // [2][128 slots][128 B]
  static constexpr uint32_t P = 4 * kBlk;       // [2][128 rows][128 B]
  static constexpr uint32_t BARS = 6 * kBlk;    // q_full, s_done, o_done
  static constexpr uint32_t TSLOT = BARS + 3 * 8;
  static constexpr uint32_t SCAL = TSLOT + 8;   // s_count etc (4 ints)
  static constexpr uint32_t RMAX = SCAL + 32;   // [2][128] row max of each column half
  static constexpr uint32_t LSUM = RMAX;        // [2][128] row sums (after the tile loop)
  static constexpr uint32_t INFO = RMAX + 1024; // [QB][kSlots] float bias of the tile
};

// Swizzled byte offset of 16-byte chunk `ch` (0..15) of 128-element row `r`
// in a K-major tile made of two 64-element blocks.
__device__ __forceinline__ uint32_t sw_off(int r, int ch) {
  return (uint32_t)((ch >> 3) * kBlk + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

template <int QB>
__global__ void __launch_bounds__(kThreads) attn_fwd_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __nv_bfloat16* __restrict__ kv,
    const int32_t* __restrict__ idx, const float* __restrict__ sink, float scale,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int sq, int H, int n_c, int ratio,
    int window, int K, int* __restrict__ status, const int32_t* __restrict__ doc, int tb, int te) {
  constexpr int NW = (QB + 3) / 4;               // u64 count words per block id
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + Layout::BARS);
  uint64_t* bar_s = bar_q + 1;
  uint64_t* bar_o = bar_q + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::TSLOT);
  int* scal = reinterpret_cast<int*>(sm + Layout::SCAL);
  float* rmax = reinterpret_cast<float*>(sm + Layout::RMAX);
  float* lsum = reinterpret_cast<float*>(sm + Layout::LSUM);
  float* bias = reinterpret_cast<float*>(sm + Layout::INFO);                 // [QB][kSlots]
  uint64_t* cnt = reinterpret_cast<uint64_t*>(bias + QB * kSlots);           // [n_c][NW]
  int* ulist = reinterpret_cast<int*>(cnt + (size_t)n_c * NW);                // [n_c]
  int* wsum = ulist + n_c;                                                    // [8] scan scratch

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bi, xb;
  heavy_first_block((te - tb + QB - 1) / QB, &bi, &xb);
  const int t0 = tb + xb * QB;       // rows t0 .. t0+QB-1 below te are this block's queries
  const int n_kv = sq + n_c;
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * kD;

  // ---- set-up: barriers, TMEM, Q tile (TMA) ---------------------------------
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  for (int e = tid; e < n_c * NW; e += kThreads) cnt[e] = 0ull;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  // Test hook (csa_debug_arm_fault): with kSiteFwdQ armed the Q tile is never
  // requested, so the bounded wait on it runs out with nothing in flight;
  // with kSiteFwdUnion armed the union-size check below trips.
  const int armed = armed_fault(status);
  if (tid == 0 && armed != kSiteFwdQ) {
    mbar_expect_tx(bar_q, 2 * kBlk);
    const int row0 = (bi * sq + t0) * H;
    tma_load_2d(sm + Layout::Q, &tmap_q, bar_q, 0, row0);
    tma_load_2d(sm + Layout::Q + kBlk, &tmap_q, bar_q, 64, row0);
  }

  // ---- union of the block's selected compressed blocks ----------------------
  const int t_last = min(t0 + QB, te) - 1;
  const int nu = build_union<QB, kThreads>(idx, bi, sq, K, t0, te, ratio, n_c, cnt, ulist, wsum,
                                           scal);
  const int win0 = max(0, t0 - window + 1);
  const int nwin = t_last - win0 + 1;
  const int S_total = nwin + nu;
  const int ntiles = (S_total + kSlots - 1) / kSlots;

  // ---- per-thread state: one TMEM lane (row) and one half of its columns ----
  const int qd = warp & 3, hf = warp >> 2;
  const int r = qd * 32 + lane;              // row = TMEM lane
  const int q = r / H, h = r % H;
  const int t = t0 + q;
  const bool row_ok = t < te;
  const float sc2 = scale * kLog2e;
  float m_run = (row_ok && sink != nullptr) ? sink[h] * kLog2e : -INFINITY;
  // the sink's unit mass is carried by the partial sum of column half 0
  float l_run = (row_ok && sink != nullptr && hf == 0) ? 1.f : 0.f;
  const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
  const uint32_t tS = tmem + lane_base + hf * 64;          // this thread's 64 score columns
  const uint32_t tO = tmem + lane_base + 128 + hf * 64;    // this thread's 64 output columns
  const float* biasq = bias + q * kSlots + hf * 64;
  // Every wait below is bounded, and every abort decision is made by the
  // whole CTA (__syncthreads_and), so no thread leaves a barrier loop alone.
  bool ok = __syncthreads_and(mbar_wait(bar_q, 0));
  int site = ok ? 0 : kSiteFwdQ;
  int code = kDevTimeout;
  // Device check: the union is a subset of the block's visible blocks, so it
  // fits the n_c-entry list the shared memory was sized for (the decision is
  // CTA-uniform: nu and the limit are the same in every thread).
  const int union_limit = armed == kSiteFwdUnion ? -1 : n_c;
  if (ok && nu > union_limit) {
    ok = false;
    site = kSiteFwdUnion;
    code = kDevCheck;
  }

  for (int it = 0; it < ntiles && ok; ++it) {
    if (it > 0) {
      ok = __syncthreads_and(mbar_wait(bar_o, (it - 1) & 1));
      if (!ok) { site = kSiteFwdO; break; }
    }
    const int sbase = it * kSlots;
    // gather KV rows of slots [sbase, sbase+128) into the swizzled tile; the
    // padding slots past the union are zero-filled rather than all reading
    // one row (which would pile every CTA's requests onto one L2 line)
    for (int c = tid; c < kSlots * 16; c += kThreads) {
      const int rr = c >> 4, ch = c & 15;
      const int s = sbase + rr;
      if (s >= S_total) {
        *reinterpret_cast<uint4*>(sm + Layout::KV + sw_off(rr, ch)) = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      const int row = s < nwin ? win0 + s : sq + ulist[s - nwin];
      cp_async_16(sm + Layout::KV + sw_off(rr, ch), kv_b + (long long)row * kD + ch * 8);
    }
    // per-query logit bias of the tile's slots: 0, log2(multiplicity) or -inf
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
      bias[e] = bv;
    }
    cp_async_wait_all_();
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0) {
      fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32_major(kRows, kSlots, 0, 0);
      const uint32_t qa = smem_addr(sm + Layout::Q), kva = smem_addr(sm + Layout::KV);
#pragma unroll
      for (int k = 0; k < kD / 16; ++k) {
        const uint32_t off = (k >> 2) * kBlk + (k & 3) * 32;
        mma_bf16_ss(tmem, sw128_desc(qa + off), sw128_desc(kva + off), idesc, k > 0 ? 1u : 0u);
      }
      mma_commit(bar_s);
    }
    ok = __syncthreads_and(mbar_wait(bar_s, it & 1));
    if (!ok) { site = kSiteFwdS; break; }
    fence_after();
    // ---- softmax: one optimistic pass against the running max -----------------
    // P = exp2(x - m_run) is written while the tile max is tracked; only rows
    // whose max grew by more than 2^8 (or had no reference yet) redo their P.
    unsigned char* pbuf = sm + Layout::P;
    const float mref = m_run == -INFINITY ? 0.f : m_run;
    float mt = -INFINITY, psum = 0.f;
#pragma unroll
    for (int c4 = 0; c4 < 2; ++c4) {
      uint32_t v[32];
      tmem_ld32_wait(tS + c4 * 32, v);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // masked slots: x = -inf and 2^-inf = 0
          const float x = fmaf(__uint_as_float(v[c8 * 8 + e]), sc2, biasq[c4 * 32 + c8 * 8 + e]);
          mt = fmaxf(mt, x);
          p[e] = ex2(x - mref);
          psum += p[e];
        }
        uint4 u;
        u.x = pack_bf16x2(p[0], p[1]);
        u.y = pack_bf16x2(p[2], p[3]);
        u.z = pack_bf16x2(p[4], p[5]);
        u.w = pack_bf16x2(p[6], p[7]);
        *reinterpret_cast<uint4*>(pbuf + sw_off(r, hf * 8 + c4 * 4 + c8)) = u;
      }
    }
    rmax[hf * kRows + r] = mt;
    __syncthreads();
    mt = fmaxf(mt, rmax[(hf ^ 1) * kRows + r]);
    const bool upd = mt > m_run + kRescale || (m_run == -INFINITY && mt != -INFINITY);
    // TMEM accesses are .sync.aligned: the whole warp takes part whenever one
    // of its rows needs them
    if (__any_sync(0xffffffffu, upd)) {
      const float alpha = upd ? ex2(m_run - mt) : 1.f;     // 0 when m_run = -inf
      // rescale this thread's half of the O row (no MMA is in flight on O here)
      if (it > 0 && __any_sync(0xffffffffu, upd && m_run != -INFINITY)) {
        const float f = (upd && m_run != -INFINITY) ? alpha : 1.f;
#pragma unroll
        for (int c4 = 0; c4 < 2; ++c4) {
          uint32_t v[32];
          tmem_ld32_wait(tO + c4 * 32, v);
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * f);
          CSA_TMEM_ST32(tO + c4 * 32, v);
        }
        tmem_wait_st();
      }
      if (upd) {
        l_run *= alpha;
        m_run = mt;
      }
      // redo P against the new max for the rows that moved it
      float psum2 = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 2; ++c4) {
        uint32_t v[32];
        tmem_ld32_wait(tS + c4 * 32, v);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float x = fmaf(__uint_as_float(v[c8 * 8 + e]), sc2, biasq[c4 * 32 + c8 * 8 + e]);
            p[e] = ex2(x - m_run);
            psum2 += p[e];
          }
          if (upd) {
            uint4 u;
            u.x = pack_bf16x2(p[0], p[1]);
            u.y = pack_bf16x2(p[2], p[3]);
            u.z = pack_bf16x2(p[4], p[5]);
            u.w = pack_bf16x2(p[6], p[7]);
            *reinterpret_cast<uint4*>(pbuf + sw_off(r, hf * 8 + c4 * 4 + c8)) = u;
          }
        }
      }
      if (upd) psum = psum2;
    }
    l_run += psum;
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0) {
      fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32_major(kRows, kD, 0, 1);
      const uint32_t pa = smem_addr(sm + Layout::P), kva = smem_addr(sm + Layout::KV);
#pragma unroll
      for (int k = 0; k < kSlots / 16; ++k) {
        const uint64_t a = sw128_desc(pa + (k >> 2) * kBlk + (k & 3) * 32);
        const uint64_t b = sw128_desc_mn(kva + k * 16 * 128, kBlk);
        mma_bf16_ss(tmem + 128, a, b, idesc, (it > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(bar_o);
    }
  }
  if (ok && ntiles > 0) {
    ok = __syncthreads_and(mbar_wait(bar_o, (ntiles - 1) & 1));
    if (!ok) site = kSiteFwdLast;
  }
  if (!ok && tid == 0) set_status(status, code, site);
  fence_after();
  // ---- epilogue: O = O / l, LSE ------------------------------------------------
  lsum[hf * kRows + r] = l_run;
  __syncthreads();
  if (ok) {
    const float l_tot = lsum[r] + lsum[kRows + r];
    // every thread loads its TMEM half row (.sync.aligned); only valid rows store
    const float inv = row_ok ? 1.f / l_tot : 0.f;
    // O rows staged in the P buffer (free: the last PV product has completed),
    // [128 rows][256 B] with the 16-byte chunks of a row rotated by the lane
    // so that the 32 rows of a warp hit different banks, then written by one
    // bulk copy of the block's contiguous rows
    unsigned char* orow_s = sm + Layout::P + r * (kD * 2) + hf * 128;
    uint4 u[8];                                  // this thread's 8 chunks of 16 B
#pragma unroll
    for (int c4 = 0; c4 < 2; ++c4) {
      uint32_t v[32];
      tmem_ld32_wait(tO + c4 * 32, v);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint4& w = u[c4 * 4 + c8];
        w.x = pack_bf16x2(__uint_as_float(v[c8 * 8 + 0]) * inv, __uint_as_float(v[c8 * 8 + 1]) * inv);
        w.y = pack_bf16x2(__uint_as_float(v[c8 * 8 + 2]) * inv, __uint_as_float(v[c8 * 8 + 3]) * inv);
        w.z = pack_bf16x2(__uint_as_float(v[c8 * 8 + 4]) * inv, __uint_as_float(v[c8 * 8 + 5]) * inv);
        w.w = pack_bf16x2(__uint_as_float(v[c8 * 8 + 6]) * inv, __uint_as_float(v[c8 * 8 + 7]) * inv);
      }
    }
    // store chunk (c + lane) % 8 at step c (a 3-stage barrel shift keeps the
    // register indices static)
#pragma unroll
    for (int k = 1; k < 8; k <<= 1) {
      const bool rot = (lane & k) != 0;
      uint4 tmp[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) tmp[c] = rot ? u[(c + k) & 7] : u[c];
#pragma unroll
      for (int c = 0; c < 8; ++c) u[c] = tmp[c];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(orow_s + ((c + lane) & 7) * 16) = u[c];
    if (row_ok && hf == 0)
      lse[(long long)(bi * sq + t0) * H + r] = (m_run + log2f(l_tot)) * kLn2;
    fence_proxy_async_smem();
  }
  fence_before();
  __syncthreads();
  if (ok && tid == 0) {
    const int nrows = min(QB, te - t0) * H;
    bulk_store(o + (long long)(bi * sq + t0) * H * kD, sm + Layout::P, (uint32_t)nrows * kD * 2u);
    bulk_commit();
    bulk_wait_read_all();      // the copy has read the staging before the CTA exits
  }
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace atc

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

size_t attn_tc_smem(int QB, int n_c) {
  const int NW = (QB + 3) / 4;
  return 1024 + atc::Layout::INFO + (size_t)QB * atc::kSlots * 4 + (size_t)n_c * NW * 8 +
         (size_t)n_c * 4 + 64;
}
}  // namespace

// Tensor-core forward available for this shape?
bool attn_tc_supported(int H, int d, int n_c, int K) {
  if (d != 128 || !(H == 16 || H == 32 || H == 64) || K > 65535) return false;
  if (encode_fn() == nullptr) return false;
  return attn_tc_smem(128 / H, n_c) <= 200 * 1024;
}

cudaError_t launch_attn_fwd_tc(const void* q, const void* kv, const int32_t* idx,
                               const float* sink, float scale, void* o, float* lse, int b, int sq,
                               int H, int n_c, int ratio, int window, int K, int* status,
                               cudaStream_t s, const int32_t* doc, int tb, int te) {
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tq;
  const cuuint64_t dims[2] = {(cuuint64_t)atc::kD, (cuuint64_t)b * sq * H};
  const cuuint64_t strides[1] = {(cuuint64_t)atc::kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)atc::kRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int QB = 128 / H;
  const size_t smem = attn_tc_smem(QB, n_c);
  dim3 grid((unsigned)(((te - tb + QB - 1) / QB) * b));   // heaviest blocks first
#define CSA_TC_FWD(QQ)                                                                          \
  {                                                                                             \
    auto k = atc::attn_fwd_tc_kernel<QQ>;                                                       \
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);           \
    k<<<grid, atc::kThreads, smem, s>>>(tq, (const __nv_bfloat16*)kv, idx, sink, scale,       \
                                        (__nv_bfloat16*)o, lse, sq, H, n_c, ratio, window, K, \
                                        status, doc, tb, te);                                   \
    count_launches(1);                                                                          \
  }
  if (QB == 8) CSA_TC_FWD(8)
  else if (QB == 4) CSA_TC_FWD(4)
  else CSA_TC_FWD(2)
#undef CSA_TC_FWD
  return cudaGetLastError();
}

}  // namespace csa
