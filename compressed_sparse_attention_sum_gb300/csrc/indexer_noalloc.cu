// csa_indexer_topk_noalloc: the indexer + top-k for callers that cannot
// allocate device memory.
//
// csa_indexer_topk needs a caller-provided workspace for the fp32 score rows
// of the queries it is processing.  Some callers have no way to provide one:
// a plugin or custom operator running inside a host framework that owns all
// device memory and exposes no allocator to it, a serving loop that must not
// call cudaMalloc after start-up (cudaMalloc can synchronize the device and
// stall every stream), or a C caller that simply has no buffer to spare.
// This variant keeps its scratch in a fixed array in the library's own device
// memory instead, and otherwise runs the same kernels as csa_indexer_topk.
//
// The array is CSA_NOALLOC_SCRATCH_BYTES (16 MiB) per device; every GPU that
// loads the library holds it until the process exits.  Problems whose score
// rows do not fit are processed in chunks of query rows; a problem whose
// smallest chunk (128 query rows of every batch element) does not fit is
// rejected with CSA_ERR_WORKSPACE before any work is enqueued.
#include <cstddef>
#include <cstdlib>
#include <mutex>

#include "../../include/csa.h"
#include "csa_common.cuh"
#include "csa_kernels.h"

namespace csa {
bool indexer_tc_supported(int H_I, int d_I);
cudaError_t launch_indexer_scores_tc(const void* q_idx, const void* k_idx, const float* w,
                                     float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                     int d_I, int ratio, int* status, cudaStream_t s);
cudaError_t launch_indexer_scores_simt(const void* q_idx, const void* k_idx, const float* w,
                                       float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                       int d_I, int ratio, bool bf16, cudaStream_t s);
int* device_status_word();
}  // namespace csa

// The scratch itself: score rows of one chunk of queries, [b][rows][n_c] fp32.
static __device__ __align__(256) float g_noalloc_scores[CSA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kTileRows = 128;
std::mutex g_setup_mutex;
float* g_scores_ptr[kMaxDevices] = {nullptr};   // device address of the array, per device

// Host code cannot hand g_noalloc_scores to a kernel directly: on the host
// that name is only a stand-in for the device symbol.  The device address is
// looked up once per device (with that device current) and cached.
float* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scores_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scores) != cudaSuccess) return nullptr;
    g_scores_ptr[dev] = static_cast<float*>(p);
  }
  return g_scores_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" csa_status_t csa_indexer_topk_noalloc(const void* q_idx, const void* k_idx,
                                                  const float* w, int32_t* topk_idx,
                                                  float* topk_score, int b, int sq, int n_c,
                                                  int H_I, int d_I, int ratio, int topk,
                                                  csa_dtype_t dt, csa_stream_t stream) {
  if (dt != CSA_FP32 && dt != CSA_BF16) return CSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || k_idx == nullptr || w == nullptr || topk_idx == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(topk_idx) ||
      !aligned16(topk_score))
    return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || H_I < 1 || d_I < 8 || d_I % 8 != 0 || ratio < 1 || topk < 1)
    return CSA_ERR_INVALID_ARG;
  if (sq < ratio || n_c != sq / ratio) return CSA_ERR_INVALID_ARG;
  if (d_I > 256 || n_c > 16384) return CSA_ERR_UNSUPPORTED;
  // the smallest chunk must fit in the fixed scratch
  const size_t row_bytes = (size_t)b * (size_t)n_c * sizeof(float);
  if (row_bytes * kTileRows > (size_t)CSA_NOALLOC_SCRATCH_BYTES) return CSA_ERR_WORKSPACE;
  float* scratch = scratch_for_current_device();
  if (scratch == nullptr) return CSA_ERR_CUDA;

  size_t rows = (size_t)CSA_NOALLOC_SCRATCH_BYTES / row_bytes;
  rows = rows / kTileRows * kTileRows;
  if (rows > (size_t)sq) rows = (size_t)sq;
  const int K = topk < n_c ? topk : n_c;
  const char* cc = getenv("CSA_INDEXER_CUDA_CORES");
  const bool use_tc = dt == CSA_BF16 && !(cc && cc[0] == '1') &&
                      csa::indexer_tc_supported(H_I, d_I);
  cudaStream_t s = (cudaStream_t)stream;
  // Every score the select kernel reads is first written by the score kernel
  // of the same chunk, so nothing left in the array by an earlier call is ever
  // read and the array needs no clearing.
  for (int t0 = 0; t0 < sq; t0 += (int)rows) {
    const int nt = (sq - t0) < (int)rows ? (sq - t0) : (int)rows;
    cudaError_t e;
    if (use_tc)
      e = csa::launch_indexer_scores_tc(q_idx, k_idx, w, scratch, t0, nt, b, sq, n_c, H_I, d_I,
                                        ratio, csa::device_status_word(), s);
    else
      e = csa::launch_indexer_scores_simt(q_idx, k_idx, w, scratch, t0, nt, b, sq, n_c, H_I, d_I,
                                          ratio, dt == CSA_BF16, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    e = csa::launch_topk_select(scratch, topk_idx, topk_score, t0, nt, b, sq, n_c, ratio, K, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  }
  return CSA_OK;
}
