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
//
// It takes no doc_ids: every batch row is one document (the candidates of
// query t are all blocks j < vis(t)).  Limits, argument checks and the chunk
// loop are those of csa_indexer_topk (indexer_host.h).
#include <cstddef>
#include <cstdlib>
#include <mutex>

#include "../../include/csa.h"
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "indexer_host.h"

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
std::mutex g_setup_mutex;
float* g_scores_ptr[kMaxDevices] = {nullptr};   // device address of the array, per device

// Host code cannot hand g_noalloc_scores to a kernel directly: on the host
// that name is only a stand-in for the device symbol.  The device address is
// looked up once per device (with that device current) and cached for the
// life of the process; the cache is not refreshed after a cudaDeviceReset of
// that device, so a caller that resets a device must not call this entry
// point on it again.
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

}  // namespace

extern "C" csa_status_t csa_indexer_topk_noalloc(const void* q_idx, const void* k_idx,
                                                  const float* w, int32_t* topk_idx,
                                                  float* topk_score, int b, int sq, int n_c,
                                                  int H_I, int d_I, int ratio, int topk,
                                                  csa_dtype_t dt, csa_stream_t stream) {
  using csa::aligned16;
  if (dt != CSA_FP32 && dt != CSA_BF16) return CSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || k_idx == nullptr || w == nullptr || topk_idx == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(topk_idx) ||
      !aligned16(topk_score))
    return CSA_ERR_INVALID_ARG;
  const csa_status_t st = csa::check_indexer_shape(b, sq, n_c, H_I, d_I, ratio, topk, 8);
  if (st != CSA_OK) return st;
  // the smallest chunk must fit in the fixed scratch
  if (csa::indexer_min_chunk_bytes(b, n_c) > (size_t)CSA_NOALLOC_SCRATCH_BYTES)
    return CSA_ERR_WORKSPACE;
  float* scratch = scratch_for_current_device();
  if (scratch == nullptr) return CSA_ERR_CUDA;

  const bool use_tc = dt == CSA_BF16 && !csa::indexer_cuda_cores_forced() &&
                      csa::indexer_tc_supported(H_I, d_I);
  int* status = csa::device_status_word();
  cudaStream_t s = (cudaStream_t)stream;
  // Every score the select kernel reads is first written by the score kernel
  // of the same chunk, so nothing left in the array by an earlier call is ever
  // read and the array needs no clearing.
  return csa::indexer_chunks(b, sq, n_c, ratio, topk, nullptr, topk_idx, topk_score, scratch,
                             (size_t)CSA_NOALLOC_SCRATCH_BYTES, s, 0, sq,
                             [&](float* ws, int t0, int nt) {
    return use_tc ? csa::launch_indexer_scores_tc(q_idx, k_idx, w, ws, t0, nt, b, sq, n_c, H_I,
                                                  d_I, ratio, status, s)
                  : csa::launch_indexer_scores_simt(q_idx, k_idx, w, ws, t0, nt, b, sq, n_c, H_I,
                                                    d_I, ratio, dt == CSA_BF16, s);
  });
}
