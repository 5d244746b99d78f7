// Indexer distillation teacher on the 5th-generation tensor cores (tcgen05 +
// TMEM), bf16, d = 128, H in {16, 32, 64}.
//
// Semantics as csa_indexer_teacher ("Refactor Deepseek v4 to use Attention
// Gym's Compressed Sparse Attention", indexer distillation; "Add unfused SBHD
// compressed sparse attention", review of the teacher normalization): for
// each valid entry s of query t's index row (block j),
//   T[s] = sum_h exp(scale q[t,h] . kv[sq + j] - lse[t,h]),
// target = T / sum_s T, with one common shift per row so that the largest
// term is 1 (it cancels in the normalization), 0 at invalid entries.
//
// A job is a block of QB = 128 / H consecutive queries, i.e. 128 (query, head)
// rows; persistent CTAs (one per SM) take the jobs heaviest first, and each
// job walks the union of the blocks its queries selected (the attention
// kernels' union) in tiles of 128 blocks.  Per tile one thread issues the transposed
// product S^T = KV Q^T (M = 128 blocks on the TMEM lanes, N = 128 rows on the
// columns, K = d) into one of two TMEM buffers, so that the next tile's
// product runs while the threads read the current one.  A thread owns one
// block (lane) and a group of 32 rows (columns): for each query in its rows
// that selected the block it forms m = max_h a_h and s = sum_h 2^(a_h - m),
// a_h = log2(e) (scale q_h . kv_j - lse_h), over the query's heads in the
// group (a query's 64 heads span two groups), and keeps (m, s) per (query,
// block, group part) in shared memory.  At the end each query's index row is
// read back in order: one pass forms the row's shift (the maximum m over its
// valid entries) and the shifted sum together (a running maximum), a second
// writes T_s / sum with T_s = s 2^(m - shift) (the parts of a 64-head query
// merged).  The next job's Q tile streams in during this step.  Every mbarrier wait is bounded; a wait that gives up
// records CSA_ERR_TIMEOUT in the device status word and the CTA skips to
// teardown.
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"
#include "attn_union.cuh"

#include <cudaTypedefs.h>

namespace csa {
namespace itc {

using namespace csa::umma;

constexpr int kRows = 128;
constexpr int kSlots = 128;
constexpr int kD = 128;
constexpr int kThreads = 512;                   // 16 warps: TMEM lane quarter x column group
constexpr uint32_t kTmemCols = 256;            // two S^T buffers of 128 columns
constexpr uint32_t kBlk = kRows * 128;          // 16 KB: 128 lines of 128 B

struct Layout {
  static constexpr uint32_t Q = 0;              // [2][128 rows][128 B] K-major
  static constexpr uint32_t KV = 2 * kBlk;      // two buffers of [2][128 blocks][128 B]
  static constexpr uint32_t BARS = 6 * kBlk;    // q, s[2]
  static constexpr uint32_t TSLOT = BARS + 3 * 8;
  static constexpr uint32_t SCAL = TSLOT + 8;
  static constexpr uint32_t LSE2 = SCAL + 64;   // [128] floats
  static constexpr uint32_t RED = LSE2 + 512;   // [2][16] floats: per-warp max, sum
  static constexpr uint32_t WSUM = RED + 128;   // [16] ints (union compaction)
  static constexpr uint32_t DYN = WSUM + 64;    // cnt, ulist, PM, PS
};

__device__ __forceinline__ uint32_t sw_off(int r, int ch) {
  return (uint32_t)((ch >> 3) * kBlk + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1) teacher_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __nv_bfloat16* __restrict__ kv,
    const int32_t* __restrict__ idx, const float* __restrict__ lse, float scale,
    float* __restrict__ target, int sq, int n_c, int ratio, int K, int* __restrict__ status,
    int njobs) {
  constexpr int QB = kRows / H;                 // queries per CTA
  constexpr int NW = (QB + 3) / 4;              // u64 count words per block
  constexpr int HS = H < 32 ? H : 32;           // heads of one query in a column group
  constexpr int NSEG = 32 / HS;                 // queries in a column group
  constexpr int P = H > 32 ? H / 32 : 1;        // column groups per query
  constexpr int WPQ = 16 / QB;                  // warps per query in the final pass
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + Layout::BARS);
  uint64_t* bar_s = bar_q + 1;                  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Layout::TSLOT);
  int* scal = reinterpret_cast<int*>(sm + Layout::SCAL);
  float* lse2 = reinterpret_cast<float*>(sm + Layout::LSE2);
  float* red = reinterpret_cast<float*>(sm + Layout::RED);
  int* wsum = reinterpret_cast<int*>(sm + Layout::WSUM);
  uint64_t* cnt = reinterpret_cast<uint64_t*>(sm + Layout::DYN);     // [n_c][NW]
  int* ulist = reinterpret_cast<int*>(cnt + (size_t)n_c * NW);       // [n_c]
  float* PM = reinterpret_cast<float*>(ulist + n_c);                 // [QB * P][n_c]
  float* PS = PM + (size_t)QB * P * n_c;                             // [QB * P][n_c]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = (sq + QB - 1) / QB;
  const int nb = njobs / nblk;                  // batch elements
  const int n_kv = sq + n_c;
  // Persistent CTAs: job j is query block nblk-1-j/nb of batch element j%nb
  // (heaviest first), dealt in sweeps of G jobs whose order alternates
  const int G = (int)gridDim.x;
  auto job_of = [&](int sweep) -> int {
    const int c = (sweep & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const int j = sweep * G + c;
    return j < njobs ? j : -1;
  };
  auto load_q = [&](int j) {                    // thread 0: job j's Q tile
    const int row0 = ((j % nb) * sq + (nblk - 1 - j / nb) * QB) * H;
    mbar_expect_tx(bar_q, 2 * kBlk);
    tma_load_2d(sm + Layout::Q, &tmap_q, bar_q, 0, row0);
    tma_load_2d(sm + Layout::Q + kBlk, &tmap_q, bar_q, 64, row0);
  };

  // ---- set-up (once per CTA): barriers, TMEM -------------------------------------
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_s + 1, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const int qd = warp & 3, cg = warp >> 2;      // lane quarter, column group
  const int r = qd * 32 + lane;                 // this thread's block within a tile
  const float sc2 = scale * kLog2e;
  uint32_t n_q = 0, n_s0 = 0, n_s1 = 0;         // completed phases, carried across jobs
  bool ok = true;
  int site = 0;
  int job = job_of(0);
  if (tid == 0 && job >= 0) load_q(job);

  for (int sweep = 0; job >= 0; ++sweep) {
  const int bi = job % nb, t0 = (nblk - 1 - job / nb) * QB;
  const __nv_bfloat16* kv_b = kv + (long long)bi * n_kv * kD;
  const int next = job_of(sweep + 1);
  for (int e = tid; e < n_c * NW; e += kThreads) cnt[e] = 0ull;
  if (tid < kRows) {
    const int t = t0 + tid / H;
    lse2[tid] = t < sq ? lse[((long long)bi * sq + t0) * H + tid] * kLog2e : INFINITY;
  }
  __syncthreads();

  // ---- union of the block's selected compressed blocks --------------------------
  const int nu = build_union<QB, kThreads>(idx, bi, sq, K, t0, sq, ratio, n_c, cnt, ulist, wsum,
                                           scal);
  const int ntiles = (nu + kSlots - 1) / kSlots;

  // gather union tile `it` (compressed rows) into KV buffer (it & 1)
  auto stage_tile = [&](int it) {
    const int sbase = it * kSlots;
    unsigned char* dst = sm + Layout::KV + (it & 1) * 2 * kBlk;
    for (int c = tid; c < kSlots * 16; c += kThreads) {
      const int rr = c >> 4, ch = c & 15;
      if (sbase + rr >= nu) {             // padding: zeros
        *reinterpret_cast<uint4*>(dst + sw_off(rr, ch)) = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      cp_async_16(dst + sw_off(rr, ch),
                  kv_b + (long long)(sq + ulist[sbase + rr]) * kD + ch * 8);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // S^T of tile `it` into TMEM buffer (it & 1): A = KV tile (M = blocks),
  // B = Q tile (N = rows), both K-major
  auto issue = [&](int it) {
    constexpr uint32_t idesc = idesc_bf16_f32_major(kSlots, kRows, 0, 0);
    const uint32_t ka = smem_addr(sm + Layout::KV + (it & 1) * 2 * kBlk);
    const uint32_t qa = smem_addr(sm + Layout::Q);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k) {
      const uint32_t off = (k >> 2) * kBlk + (k & 3) * 32;
      mma_bf16_ss(tmem + (it & 1) * 128, sw128_desc(ka + off), sw128_desc(qa + off), idesc,
                  k > 0 ? 1u : 0u);
    }
    mma_commit(&bar_s[it & 1]);
  };

  ok = __syncthreads_and(mbar_wait(bar_q, n_q & 1));
  if (!ok) { site = kSiteTeacherQ; break; }
  ++n_q;
  if (ntiles > 0) {
    stage_tile(0);
    if (ntiles > 1) {
      stage_tile(1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    if (tid == 0) {
      fence_after();
      issue(0);
    }
  }
  for (int it = 0; it < ntiles && ok; ++it) {
    if (it + 1 < ntiles) {
      // tile it+1 has arrived: its product goes into the other buffer
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      fence_proxy_async_smem();
      fence_before();
      __syncthreads();
      if (tid == 0) {
        fence_after();
        issue(it + 1);
      }
    }
    // per-warp wait: a warp starts its sums as soon as the scores are there,
    // not after the issuing thread has handed the next tile's product over
    const bool got =
        __all_sync(0xffffffffu, mbar_wait(&bar_s[it & 1], (((it & 1) ? n_s1 : n_s0) + (it >> 1)) & 1));
    if (got) {
      fence_after();
      uint32_t v[32];
      tmem_ld32_wait(tmem + ((uint32_t)(qd * 32) << 16) + (it & 1) * 128 + cg * 32, v);
      const int u = it * kSlots + r;
      if (u < nu) {
        const int j = ulist[u];
#pragma unroll
        for (int sg = 0; sg < NSEG; ++sg) {
          const int row0 = cg * 32 + sg * HS;
          const int q = row0 / H;
          const uint32_t c = (uint32_t)(cnt[j * NW + (q >> 2)] >> (16 * (q & 3))) & 0xFFFFu;
          if (c == 0u) continue;                // the query did not select this block
          float a[HS], m = -INFINITY;
#pragma unroll
          for (int h = 0; h < HS; ++h) {
            a[h] = fmaf(__uint_as_float(v[sg * HS + h]), sc2, -lse2[row0 + h]);
            m = fmaxf(m, a[h]);
          }
          float s = 0.f;
#pragma unroll
          for (int h = 0; h < HS; ++h) s += ex2(a[h] - m);
          const int part = (row0 % H) / 32;
          PM[(size_t)(q * P + part) * n_c + j] = m;
          PS[(size_t)(q * P + part) * n_c + j] = s;
        }
      }
    }
    fence_before();
    // every thread is done with this tile's TMEM buffer; its KV buffer was
    // released when the product completed: stage tile it+2 there
    ok = !__syncthreads_or(!got);
    if (!ok) { site = kSiteTeacherS; break; }
    if (it + 2 < ntiles) stage_tile(it + 2);
  }
  if (!ok) break;
  n_s0 += (ntiles + 1) / 2;
  n_s1 += ntiles / 2;
  // every product of this job has completed (its last wait above): the next
  // job's Q tile streams in under the normalization and the next union
  if (tid == 0 && next >= 0) load_q(next);

  // ---- per query: the row shift, the terms and the L1 normalization --------------
  {
    const int q = warp / WPQ, wq = warp % WPQ;
    const int t = t0 + q;
    const int tl = wq * 32 + lane, nthr = WPQ * 32;
    const int vis = min((t + 1) / ratio, n_c);
    const int32_t* ir = idx + ((long long)bi * sq + t) * K;
    auto term = [&](int k, float* m_out) -> float {   // (m, s) of entry k, parts merged
      const int j = ir[k];
      if (j < 0 || j >= vis) return -1.f;
      float m = PM[(size_t)(q * P) * n_c + j], s = PS[(size_t)(q * P) * n_c + j];
#pragma unroll
      for (int p = 1; p < P; ++p) {
        const float m2 = PM[(size_t)(q * P + p) * n_c + j], s2 = PS[(size_t)(q * P + p) * n_c + j];
        const float mm = fmaxf(m, m2);
        s = s * ex2(m - mm) + s2 * ex2(m2 - mm);
        m = mm;
      }
      *m_out = m;
      return s;
    };
    // one pass: the running (max, shifted sum) of the row's terms, merged
    // across the query's threads
    float mx = -INFINITY, tot = 0.f;
    if (t < sq)
      for (int k = tl; k < K; k += nthr) {
        float m;
        const float s = term(k, &m);
        if (s < 0.f) continue;
        if (m > mx) {
          tot = tot * ex2(mx - m) + s;
          mx = m;
        } else {
          tot += s * ex2(m - mx);
        }
      }
    auto merge = [](float& M, float& S, float m2, float s2) {
      const float mm = fmaxf(M, m2);
      if (mm == -INFINITY) return;              // both empty
      S = S * ex2(M - mm) + s2 * ex2(m2 - mm);
      M = mm;
    };
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mx, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, tot, o);
      merge(mx, tot, m2, s2);
    }
    if (lane == 0) {
      red[warp] = mx;
      red[16 + warp] = tot;
    }
    __syncthreads();
    mx = -INFINITY;
    tot = 0.f;
    for (int w = 0; w < WPQ; ++w) merge(mx, tot, red[q * WPQ + w], red[16 + q * WPQ + w]);
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    if (t < sq) {
      float* out = target + ((long long)bi * sq + t) * K;
      for (int k = tl; k < K; k += nthr) {
        float m;
        const float s = term(k, &m);
        out[k] = s >= 0.f ? s * ex2(m - mx) * inv : 0.f;
      }
    }
  }
  // this job's shared-memory reads are done before the next job's writes
  __syncthreads();
  job = next;
  }  // jobs

  asm volatile("cp.async.wait_all;" ::: "memory");    // no copy in flight past this point
  // a failed wait for the prefetched tiles may leave them in flight (every
  // other wait precedes the next prefetch): wait for them once more (bounded)
  if (site == kSiteTeacherQ && tid == 0) mbar_wait(bar_q, n_q & 1);
  if (!ok && tid == 0) set_status(status, kDevTimeout, site);
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace itc

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_teacher() {
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

size_t teacher_tc_smem(int H, int n_c) {
  const int QB = itc::kRows / H, NW = (QB + 3) / 4, P = H > 32 ? H / 32 : 1;
  return 1024 + itc::Layout::DYN + (size_t)n_c * NW * 8 + (size_t)n_c * 4 +
         (size_t)2 * QB * P * n_c * 4;
}
}  // namespace

bool indexer_teacher_tc_supported(int H, int d, int n_c, int K) {
  if (d != itc::kD || !(H == 16 || H == 32 || H == 64) || K > 65535) return false;
  if (encode_fn_teacher() == nullptr) return false;
  return teacher_tc_smem(H, n_c) <= 227 * 1024;
}

cudaError_t launch_indexer_teacher_tc(const void* q, const void* kv, const int32_t* idx,
                                      const float* lse, float scale, float* target, int b, int sq,
                                      int H, int n_c, int ratio, int K, int* status,
                                      cudaStream_t s) {
  auto encode = encode_fn_teacher();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tq;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)itc::kD, (cuuint64_t)b * sq * H};
    const cuuint64_t strides[1] = {(cuuint64_t)itc::kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)itc::kRows};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int QB = itc::kRows / H;
  const size_t smem = teacher_tc_smem(H, n_c);
  const int njobs = ((sq + QB - 1) / QB) * b;
  int dev = 0, n_sm = 0;                        // persistent CTAs: one per SM
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1)
    return cudaErrorInvalidValue;
  dim3 grid((unsigned)(njobs < n_sm ? njobs : n_sm));
#define CSA_TEACH_TC(HH)                                                                       \
  {                                                                                            \
    auto k = itc::teacher_tc_kernel<HH>;                                                       \
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                         (int)smem);                                           \
    if (e != cudaSuccess) return e;                                                            \
    k<<<grid, itc::kThreads, smem, s>>>(tq, (const __nv_bfloat16*)kv, idx, lse, scale, target, \
                                        sq, n_c, ratio, K, status, njobs);                     \
    count_launches(1);                                                                         \
  }
  if (H == 16) CSA_TEACH_TC(16)
  else if (H == 32) CSA_TEACH_TC(32)
  else CSA_TEACH_TC(64)
#undef CSA_TEACH_TC
  return cudaGetLastError();
}

}  // namespace csa
