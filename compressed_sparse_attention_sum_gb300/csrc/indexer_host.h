// Host-side pieces shared by the indexer entry points (csa_indexer_topk,
// csa_indexer_topk_fp8, csa_indexer_topk_noalloc): the size limits, the
// argument checks and the loop over chunks of query rows.  Keeping them in
// one place keeps the entry points in step when a limit or the chunking
// changes.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstdlib>

#include "../../include/csa.h"
#include "csa_kernels.h"

namespace csa {

constexpr int kMaxD = 512;            // attention head dim
constexpr int kMaxH = 64;             // attention heads
constexpr int kMaxNc = 16384;         // compressed blocks per batch element
constexpr int kMaxDI = 256;           // indexer head dim
constexpr int kIndexerTileRows = 128; // query rows of one score tile (the chunk granule)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes of score rows of the smallest chunk: one tile of query rows of every
// batch element, n_c fp32 scores each.
inline size_t indexer_min_chunk_bytes(int b, int n_c) {
  return (size_t)b * kIndexerTileRows * (size_t)n_c * sizeof(float);
}

// Shape checks common to the bf16/fp32 indexer entry points (pointers are
// checked by each caller, since their sets differ).
inline csa_status_t check_indexer_shape(int b, int sq, int n_c, int H_I, int d_I, int ratio,
                                        int topk, int d_I_multiple) {
  if (b < 1 || sq < 1 || H_I < 1 || d_I < d_I_multiple || d_I % d_I_multiple != 0 ||
      ratio < 1 || topk < 1)
    return CSA_ERR_INVALID_ARG;
  if (sq < ratio || n_c != sq / ratio) return CSA_ERR_INVALID_ARG;
  if (d_I > kMaxDI || n_c > kMaxNc) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

// CSA_INDEXER_CUDA_CORES=1 selects the CUDA-core score kernel even where the
// tensor-core one applies (same results up to fp32 summation order; used to
// compare the two).
inline bool indexer_cuda_cores_forced() {
  const char* cc = getenv("CSA_INDEXER_CUDA_CORES");
  return cc != nullptr && cc[0] == '1';
}

// The indexer's chunk loop: the query rows [t_begin, t_end) of every batch
// element go through the score buffer in chunks of whole 128-row tiles; per
// chunk, `score(ws, t0, nt)` fills the rows' visible scores and the per-row
// select writes their top-K.  Arguments already validated; the buffer holds
// at least indexer_min_chunk_bytes(b, n_c).
template <typename ScoreFn>
csa_status_t indexer_chunks(int b, int sq, int n_c, int ratio, int topk, const int32_t* doc_ids,
                            int32_t* topk_idx, float* topk_score, void* buf, size_t buf_bytes,
                            cudaStream_t s, int t_begin, int t_end, ScoreFn score) {
  const size_t row_bytes = (size_t)b * n_c * sizeof(float);
  const int K = topk < n_c ? topk : n_c;
  size_t rows = buf_bytes / row_bytes;
  rows = rows / kIndexerTileRows * kIndexerTileRows;
  if (rows > (size_t)(t_end - t_begin)) rows = (size_t)(t_end - t_begin);
  if (rows == 0) return CSA_OK;
  for (int t0 = t_begin; t0 < t_end; t0 += (int)rows) {
    const int nt = (t_end - t0) < (int)rows ? (t_end - t0) : (int)rows;
    if (score((float*)buf, t0, nt) != cudaSuccess) return CSA_ERR_CUDA;
    if (launch_topk_select((const float*)buf, topk_idx, topk_score, t0, nt, b, sq, n_c, ratio, K,
                           s, doc_ids) != cudaSuccess)
      return CSA_ERR_CUDA;
  }
  return CSA_OK;
}

}  // namespace csa
