// Lightning-indexer scores on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA), bf16 inputs, fp32 accumulation.
//
//   I[b,t,j] = sum_h w[b,t,h] * max(0, q_I[b,t,h,:] . k_I[b,j,:]),  j < vis(t)
//
// ("Add unfused SBHD compressed sparse attention", indexer block; "Refactor
// Deepseek v4 to use Attention Gym's Compressed Sparse Attention", indexer
// selectability j < (t+1)//ratio.)
//
// One CTA computes a tile of 128 queries x 128 compressed blocks of one batch
// element, for all indexer heads, and writes the fp32 tile to the score
// workspace that the per-row select kernel reads.  Tiles entirely above the
// causal boundary are skipped.  Roles (352 threads):
//   warp 0      TMA producer: the k_I tile once, then one q_I head tile per
//               stage of a 6-deep ring (3D tensor map over [b*sq, H_I, d_I])
//   warps 1-2   MMA issuers (warp 1 also owns TMEM): warp 1 the even heads,
//               warp 2 the odd ones; head h goes to TMEM accumulator h % 4
//               (four, so that the tensor core runs up to three heads ahead
//               of the epilogue): d_I/16 tcgen05.mma (M=128 queries, N=128
//               blocks, K=16) per head, committed to the ring's "empty"
//               barrier and to the accumulator's "full" barrier
//   warps 3-10  epilogue: tcgen05.ld of the head's accumulator (row = query =
//               TMEM lane), release of the accumulator, then
//               I += w[t,h] * max(S, 0) in registers; each warp owns one TMEM
//               lane quarter and one half of the 128 columns
// Every mbarrier wait is bounded; a wait that gives up records
// CSA_ERR_TIMEOUT in the device status word and the CTA skips to teardown.
//
// The FP8 variant (F8) takes e4m3 codes of q_I and k_I with per-row scales
// (csa_quantize_e4m3): rows of 128 bytes hold 128 codes, each MMA is
// kind::f8f6f4 with K = 32 (the same 32-byte step along a row), and since the
// scales are positive they leave the ReLU:
//   I[t,j] = sk[j] * sum_h (w[t,h] sq[t,h]) max(0, q8[t,h] . k8[j]).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "csa_common.cuh"
#include "csa_kernels.h"
#include "tcgen05.cuh"

namespace csa {

namespace tc {

using namespace csa::umma;

constexpr int kTileM = 128;     // queries per tile (TMEM lanes)
constexpr int kTileN = 128;     // compressed blocks per tile (TMEM columns per accumulator)
constexpr int kStages = 6;
constexpr int kThreads = 352;
constexpr int kEpiWarps = 8;
constexpr int kMaxHeads = 64;
constexpr int kAcc = 4;                 // TMEM accumulators (128 columns each)
constexpr uint32_t kTmemCols = kAcc * 128;
template <int DI, bool F8>
__global__ void __launch_bounds__(kThreads, 1) indexer_scores_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_ws, int ws_tma,
    const float* __restrict__ w, float* __restrict__ ws, int t0, int nt, int sq, int n_c,
    int H_I, int ratio, int* __restrict__ status, const float* __restrict__ q_scale,
    const float* __restrict__ k_scale) {
  constexpr int EPB = F8 ? 128 : 64;                  // elements per 128-byte row block
  constexpr int KB = DI / EPB;                        // 128-byte K blocks
  constexpr uint32_t kTileBytes = KB * kTileM * 128;  // one operand tile (128 rows x DI)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sB = sm;                                     // k_I tile
  unsigned char* sA = sm + kTileBytes;                        // q_I ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + kStages * kTileBytes);
  uint64_t* full = bars;                 // [kStages]
  uint64_t* empty = bars + kStages;      // [kStages]
  uint64_t* acc_full = bars + 2 * kStages;      // [kAcc]
  uint64_t* acc_empty = acc_full + kAcc;        // [kAcc]
  uint64_t* b_full = acc_empty + kAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_full + 1);
  __shared__ int s_abort;

  const int kt = blockIdx.x, qt = blockIdx.y, bi = blockIdx.z;
  const int tq0 = t0 + qt * kTileM;
  const int tq_end = min(t0 + nt, tq0 + kTileM);
  const int vis_max = min(tq_end / ratio, n_c);
  const int j0 = kt * kTileN;
  // The select kernel that follows may be scheduled now (it waits for this
  // grid's completion before reading the scores): it then takes free SMs
  // while the score tiles run instead of starting after a launch gap.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tq0 >= tq_end || j0 >= vis_max) return;   // tile above the causal boundary

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    mbar_init(b_full, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      mbar_expect_tx(b_full, kTileBytes);
      for (int kb = 0; kb < KB; ++kb)
        tma_load_2d(sB + kb * kTileM * 128, &tmap_k, b_full, kb * EPB, bi * n_c + j0);
      for (int h = 0; h < H_I; ++h) {
        const int s = h % kStages;
        const uint32_t par = ((h / kStages) & 1) ^ 1;
        if (!mbar_wait(&empty[s], par)) {
          set_status(status, kDevTimeout, kSiteIdxProducer);
          s_abort = 1;
          break;
        }
        mbar_expect_tx(&full[s], kTileBytes);
        unsigned char* dst = sA + s * kTileBytes;
        for (int kb = 0; kb < KB; ++kb)
          tma_load_3d(dst + kb * kTileM * 128, &tmap_q, &full[s], kb * EPB, h,
                      bi * sq + tq0);
      }
    }
  } else if (warp <= 2) {
    // ---------------- MMA issuers ----------------
    // tcgen05.mma holds its issuing thread until the tensor core has taken
    // the instruction, so the waits and commits of one thread would leave the
    // tensor core idle between heads: two threads (warps 1 and 2) take the
    // even and the odd heads, and one issues while the other waits.
    if (lane == 0) {
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(kTileM, kTileN) : idesc_bf16_f32(kTileM, kTileN);
      bool ok = mbar_wait(b_full, 0);
      const uint32_t b_base = smem_addr(sB);
      for (int h = warp - 1; ok && h < H_I; h += 2) {
        const int a = h % kAcc;
        const int s = h % kStages;
        if (!mbar_wait(&full[s], (h / kStages) & 1) ||
            !mbar_wait(&acc_empty[a], ((h / kAcc) & 1) ^ 1)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t a_base = smem_addr(sA + s * kTileBytes);
        const uint32_t d_tmem = tmem_base + a * kTileN;
#pragma unroll
        for (int k = 0; k < KB * 4; ++k) {              // 32-byte K steps
          const uint32_t off = (k / 4) * kTileM * 128 + (k % 4) * 32;
          if constexpr (F8)
            mma_f8_ss(d_tmem, sw128_desc(a_base + off), sw128_desc(b_base + off), idesc,
                      k > 0 ? 1u : 0u);
          else
            mma_bf16_ss(d_tmem, sw128_desc(a_base + off), sw128_desc(b_base + off), idesc,
                        k > 0 ? 1u : 0u);
        }
        mma_commit(&empty[s]);
        mma_commit(&acc_full[a]);
      }
      if (!ok) {
        set_status(status, kDevTimeout, kSiteIdxMma);
        s_abort = 1;
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int half = (warp - 3) >> 2;             // column half of the tile
    const int row = quarter * 32 + lane;          // query within the tile
    // this query's head weights: one 4-byte read per head from its own
    // H_I-float row (L1-resident after the first touch)
    const int tw = min(tq0 + row, tq_end - 1);
    const float* wrow = w + ((long long)bi * sq + tw) * H_I;
    float acc[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) acc[c] = 0.f;
    bool ok = true;
    for (int h = 0; h < H_I; ++h) {
      const int a = h % kAcc;
      // warp-uniform decision: the TMEM loads below are .sync.aligned
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[a], (h / kAcc) & 1))) {
        ok = false;
        break;
      }
      fence_after();
      uint32_t v0[32], v1[32];
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + a * kTileN + half * 64;
      tmem_ld64(taddr, v0, v1);
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
      float wv = __ldg(wrow + h);
      if constexpr (F8) wv *= __ldg(q_scale + ((long long)bi * sq + tw) * H_I + h);
      // the weighted ReLU sum as paired fma (one instruction per two columns;
      // the ReLU stays a max)
      const unsigned long long w2 = pack_f32x2(wv, wv);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        fma_f32x2(acc[c], acc[c + 1], w2, fmaxf(__uint_as_float(v0[c]), 0.f),
                  fmaxf(__uint_as_float(v0[c + 1]), 0.f));
        fma_f32x2(acc[32 + c], acc[33 + c], w2, fmaxf(__uint_as_float(v1[c]), 0.f),
                  fmaxf(__uint_as_float(v1[c + 1]), 0.f));
      }
    }
    if (!ok) {
      set_status(status, kDevTimeout, kSiteIdxEpilogue);
      s_abort = 1;
    }
    const int t = tq0 + row;
    const int jb = j0 + half * 64;
    if constexpr (F8) {
#pragma unroll
      for (int c = 0; c < 64; ++c)
        acc[c] *= jb + c < n_c ? __ldg(k_scale + (long long)bi * n_c + jb + c) : 0.f;
    }
    if (ok && ws_tma) {
      // the tile goes through the q_I ring (every head's product has
      // completed) to one TMA store, which clips the rows past the chunk and
      // the blocks past n_c; entries past a row's visible blocks are written
      // too (the select never reads them).  A row's 16-byte chunks are
      // rotated by the lane so that the warp's 32 rows hit different banks.
      float* srow = reinterpret_cast<float*>(sA) + row * kTileN + half * 64;
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {          // two groups of 8 chunks
        float4 ch[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int e = c8 * 32 + c * 4;
          ch[c] = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
        }
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
          *reinterpret_cast<float4*>(srow + c8 * 32 + ((c + lane) & 7) * 4) = ch[c];
      }
      fence_proxy_async_smem();
    } else if (ok && t < tq_end) {
      const int vis = min((t + 1) / ratio, n_c);
      float* dst = ws + ((long long)bi * nt + (t - t0)) * n_c + jb;
      if (jb + 64 <= vis && (n_c & 3) == 0) {
#pragma unroll
        for (int c = 0; c < 64; c += 4)
          *reinterpret_cast<float4*>(dst + c) =
              make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (jb + c < vis) dst[c] = acc[c];
      }
    }
  }
  fence_before();
  __syncthreads();
  if (ws_tma && threadIdx.x == 0 && !s_abort) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            &tmap_ws),
        "r"(j0), "r"(tq0 - t0), "r"(bi), "r"(smem_addr(sA))
        : "memory");
    bulk_commit();
    bulk_wait_read_all();      // the store has read the staging before the CTA exits
  }
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace tc

namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}
}  // namespace

bool indexer_tc_supported(int H_I, int d_I) {
  return (d_I == 64 || d_I == 128) && H_I >= 1 && H_I <= tc::kMaxHeads && get_encode() != nullptr;
}
bool indexer_tc_fp8_supported(int H_I, int d_I) {
  return (d_I == 128 || d_I == 256) && H_I >= 1 && H_I <= tc::kMaxHeads && get_encode() != nullptr;
}

size_t indexer_tc_smem(int d_I, bool fp8 = false) {
  const size_t tile = (size_t)(fp8 ? d_I / 128 : d_I / 64) * tc::kTileM * 128;
  return 1024 + tile * (1 + tc::kStages) + (2 * tc::kStages + 2 * tc::kAcc + 1) * 8 + 16;
}

cudaError_t launch_indexer_scores_tc(const void* q_idx, const void* k_idx, const float* w,
                                     float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                     int d_I, int ratio, int* status, cudaStream_t s,
                                     const float* q_scale, const float* k_scale) {
  const bool f8 = q_scale != nullptr;     // e4m3 codes with per-row scales
  const int eb = f8 ? 1 : 2, epb = f8 ? 128 : 64;
  const CUtensorMapDataType dtp = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  auto encode = get_encode();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tq, tk;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d_I, (cuuint64_t)H_I, (cuuint64_t)b * sq};
    const cuuint64_t strides[2] = {(cuuint64_t)d_I * eb, (cuuint64_t)H_I * d_I * eb};
    const cuuint32_t box[3] = {(cuuint32_t)epb, 1, (cuuint32_t)tc::kTileM};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tq, dtp, 3, const_cast<void*>(q_idx), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d_I, (cuuint64_t)b * n_c};
    const cuuint64_t strides[1] = {(cuuint64_t)d_I * eb};
    const cuuint32_t box[2] = {(cuuint32_t)epb, (cuuint32_t)tc::kTileN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tk, dtp, 2, const_cast<void*>(k_idx), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the score tiles leave by TMA when the workspace rows suit a tensor map
  // (16-byte row stride and base)
  CUtensorMap tws;
  int ws_tma = 0;
  if ((n_c & 3) == 0 && (reinterpret_cast<uintptr_t>(ws) & 15) == 0) {
    // [b][nt rows][n_c]: a partial query tile is clipped at its own batch
    // element's rows
    const cuuint64_t dims[3] = {(cuuint64_t)n_c, (cuuint64_t)nt, (cuuint64_t)b};
    const cuuint64_t strides[2] = {(cuuint64_t)n_c * 4, (cuuint64_t)nt * n_c * 4};
    const cuuint32_t box[3] = {(cuuint32_t)tc::kTileN, (cuuint32_t)tc::kTileM, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    ws_tma = encode(&tws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
             CUDA_SUCCESS;
  }
  if (!ws_tma) memset(&tws, 0, sizeof(tws));
  const size_t smem = indexer_tc_smem(d_I, f8);
  dim3 grid((unsigned)((n_c + tc::kTileN - 1) / tc::kTileN),
            (unsigned)((nt + tc::kTileM - 1) / tc::kTileM), (unsigned)b);
#define CSA_IDX_TC(DD, FF)                                                                      \
  {                                                                                             \
    auto k = tc::indexer_scores_tc_kernel<DD, FF>;                                              \
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);           \
    k<<<grid, tc::kThreads, smem, s>>>(tq, tk, tws, ws_tma, w, ws, t0, nt, sq, n_c, H_I,      \
                                       ratio, status,                                          \
                                       q_scale, k_scale);                                       \
    count_launches(1);                                                                          \
  }
  if (f8) {
    if (d_I == 256) CSA_IDX_TC(256, true)
    else CSA_IDX_TC(128, true)
  } else {
    if (d_I == 128) CSA_IDX_TC(128, false)
    else CSA_IDX_TC(64, false)
  }
#undef CSA_IDX_TC
  return cudaGetLastError();
}

cudaError_t launch_indexer_scores_tc(const void* q_idx, const void* k_idx, const float* w,
                                     float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                     int d_I, int ratio, int* status, cudaStream_t s) {
  return launch_indexer_scores_tc(q_idx, k_idx, w, ws, t0, nt, b, sq, n_c, H_I, d_I, ratio,
                                  status, s, nullptr, nullptr);
}

}  // namespace csa
