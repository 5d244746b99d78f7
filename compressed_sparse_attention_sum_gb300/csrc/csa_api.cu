// C ABI entry points of the CSA library: argument validation, dispatch to the
// kernels, and the chunk loop of the indexer.  Every check runs before the
// first CUDA call, so a rejected call leaves the device untouched.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/csa.h"
#include "csa_common.cuh"
#include "csa_kernels.h"
#include "indexer_host.h"

namespace csa {
// kernels defined in the other translation units
cudaError_t launch_indexer_scores_simt(const void* q_idx, const void* k_idx, const float* w,
                                       float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                       int d_I, int ratio, bool bf16, cudaStream_t s);
bool indexer_tc_supported(int H_I, int d_I);
cudaError_t launch_indexer_scores_tc(const void* q_idx, const void* k_idx, const float* w,
                                     float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                     int d_I, int ratio, int* status, cudaStream_t s);
bool indexer_tc_fp8_supported(int H_I, int d_I);
cudaError_t launch_indexer_scores_tc(const void* q_idx, const void* k_idx, const float* w,
                                     float* ws, int t0, int nt, int b, int sq, int n_c, int H_I,
                                     int d_I, int ratio, int* status, cudaStream_t s,
                                     const float* q_scale, const float* k_scale);
cudaError_t launch_indexer_scores_simt_fp8(const uint8_t* q8, const float* q_scale,
                                           const uint8_t* k8, const float* k_scale,
                                           const float* w, float* ws, int t0, int nt, int b,
                                           int sq, int n_c, int H_I, int d_I, int ratio,
                                           cudaStream_t s);
cudaError_t launch_quantize_e4m3(const void* x, long long rows, int d, bool bf16, uint8_t* out,
                                 float* scale, cudaStream_t s);
bool attn_mma_supported(int H, int d, int window, int K);
bool attn_tc512_supported(int H, int d, int window, int Kl);
bool indexer_teacher_tc_supported(int H, int d, int n_c, int K);
cudaError_t launch_indexer_teacher_tc(const void* q, const void* kv, const int32_t* idx,
                                      const float* lse, float scale, float* target, int b, int sq,
                                      int H, int n_c, int ratio, int K, int* status,
                                      cudaStream_t s);
bool attn_tc512_bwd_supported(int H, int d, int window, int Kl);
cudaError_t launch_attn_bwd_tc512(const void* q, const void* kv, const int32_t* idx,
                                  const float* sink, float scale, const float* lse,
                                  const void* dO, float* dq, float* dkv, float* dsink, int b,
                                  int sq, int n_c, int ratio, int window, int K, int* status,
                                  cudaStream_t s, const int32_t* doc, int tb, int te);
cudaError_t launch_attn_fwd_tc512(const void* q, const void* kv, const int32_t* idx,
                                  const float* sink, float scale, void* o, float* lse, int b,
                                  int sq, int n_c, int ratio, int window, int K, int* status,
                                  cudaStream_t s, const int32_t* doc, int tb, int te);
bool attn_tc_supported(int H, int d, int n_c, int K);
bool attn_tc_bwd_supported(int H, int d, int n_c, int K);
cudaError_t launch_attn_bwd_tc(const void* q, const void* kv, const int32_t* idx,
                               const float* sink, float scale, const void* o, const float* lse,
                               const void* dO,
                               float* dq, float* dkv, float* dsink, int b, int sq, int H, int n_c,
                               int ratio, int window, int K, int* status, cudaStream_t s,
                               const int32_t* doc, int tb, int te);
cudaError_t launch_attn_fwd_tc(const void* q, const void* kv, const int32_t* idx,
                               const float* sink, float scale, void* o, float* lse, int b, int sq,
                               int H, int n_c, int ratio, int window, int K, int* status,
                               cudaStream_t s, const int32_t* doc, int tb, int te);
cudaError_t launch_attn_fwd_mma(const void* q, const void* kv, const int32_t* idx,
                                const float* sink, float scale, void* o, float* lse, int b, int sq,
                                int H, int d, int n_c, int ratio, int window, int K,
                                cudaStream_t s, const int32_t* doc, int tb, int te);
cudaError_t launch_attn_bwd_mma(const void* q, const void* kv, const int32_t* idx,
                                const float* sink, float scale, const void* o, const float* lse,
                                const void* dO, float* dq, float* dkv, float* dsink, int b, int sq,
                                int H, int d, int n_c, int ratio, int window, int K,
                                cudaStream_t s, const int32_t* doc, int tb, int te);
cudaError_t launch_attn_fwd_simt(const void* q, const void* kv, const int32_t* idx,
                                 const float* sink, float scale, void* o, float* lse, int b,
                                 int sq, int H, int d, int n_c, int ratio, int window, int K,
                                 bool bf16, cudaStream_t s, const int32_t* doc, int tb, int te);
cudaError_t launch_attn_bwd_simt(const void* q, const void* kv, const int32_t* idx,
                                 const float* sink, float scale, const void* o, const float* lse,
                                 const void* dO, float* dq, float* dkv, float* dsink, int b,
                                 int sq, int H, int d, int n_c, int ratio, int window, int K,
                                 bool bf16, cudaStream_t s, const int32_t* doc, int tb, int te);
bool indexer_teacher_mma_ok(int H, int d);
bool indexer_loss_mma_ok(int H_I, int d_I);
size_t indexer_teacher_smem(bool mma, int H, int d, int K);
size_t indexer_loss_smem(bool mma, int H_I, int d_I, int K);
cudaError_t launch_indexer_teacher(const void* q, const void* kv, const int32_t* idx,
                                   const float* lse, float scale, float* target, int b, int sq,
                                   int H, int d, int n_c, int ratio, int K, bool bf16,
                                   cudaStream_t s);
cudaError_t launch_indexer_loss(const void* q_I, const void* k_I, const float* w,
                                const int32_t* idx, const float* target, float* loss, float* dq_I,
                                float* dk_I, float* dw, int b, int sq, int H_I, int d_I, int n_c,
                                int ratio, int K, bool bf16, cudaStream_t s);
bool indexer_loss_tc_supported(int H_I, int d_I, int n_c);
cudaError_t launch_indexer_loss_tc(const void* q_I, const void* k_I, const float* w,
                                   const int32_t* idx, const float* target, float* loss,
                                   float* dq_I, float* dk_I, float* dw, int b, int sq, int H_I,
                                   int n_c, int ratio, int K, int* status, cudaStream_t s);
}  // namespace csa

#include <atomic>

namespace csa {
static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n); }
}  // namespace csa

// Device status word (one per device that loads the library): [0] the first
// error code, [1] its site, [2] the site of a faked failure armed by
// csa_debug_arm_fault (0 = none), [3] unused.
static __device__ int g_csa_device_status[4] = {0, 0, 0, 0};

namespace {

constexpr size_t kDefaultIndexerWorkspace = 128ull << 20;  // stays resident in L2
using csa::aligned16;
using csa::kMaxD;
using csa::kMaxDI;
using csa::kMaxH;
using csa::kMaxNc;

// Device address of the current device's status word.  Host code cannot hand
// g_csa_device_status to a kernel (on the host the name is only a stand-in
// for the device symbol), so the address is looked up once per device, with
// that device current, and cached.  The cache is guarded: two host threads
// may make their first call at the same time.  It is not refreshed after a
// cudaDeviceReset of that device.
std::mutex g_status_mutex;
int* g_status_ptrs[64] = {nullptr};

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mutex);
  if (g_status_ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_csa_device_status) != cudaSuccess) return nullptr;
    g_status_ptrs[dev] = static_cast<int*>(p);
  }
  return g_status_ptrs[dev];
}

}  // namespace

namespace csa {
// Device address of the status word of the current device (for the other
// translation units of the library).
int* device_status_word() { return device_status_ptr(); }
}  // namespace csa

namespace {

csa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

bool valid_dtype(csa_dtype_t dt) { return dt == CSA_FP32 || dt == CSA_BF16; }

// The query rows [tb, te) of every batch element (0 <= tb < te <= sq).
csa_status_t check_rows(int sq, int t_begin, int t_end) {
  return (t_begin < 0 || t_end > sq || t_begin >= t_end) ? CSA_ERR_INVALID_ARG : CSA_OK;
}

// Shared validation of the attention calls.
csa_status_t check_attn(const void* q, const void* kv_full, const int32_t* idx, float scale,
                        int b, int sq, int H, int d, int n_c, int ratio, int window, int K,
                        csa_dtype_t dt) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (q == nullptr || kv_full == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_full) || !aligned16(idx)) return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || H < 1 || d < 8 || d % 8 != 0 || ratio < 1 || window < 1)
    return CSA_ERR_INVALID_ARG;
  if (sq < ratio || n_c != sq / ratio) return CSA_ERR_INVALID_ARG;
  if (idx != nullptr && K < 1) return CSA_ERR_INVALID_ARG;
  if (!(scale == scale)) return CSA_ERR_INVALID_ARG;
  if (d > kMaxD || H > kMaxH || n_c > kMaxNc) return CSA_ERR_UNSUPPORTED;
  if ((size_t)(window + (idx ? K : n_c)) > 200000) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

}  // namespace

extern "C" {

const char* csa_status_string(int status) {
  switch (status) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_ARG: return "CSA_ERR_INVALID_ARG: invalid pointer, alignment or size";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: shape or dtype not implemented";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA: a CUDA call or launch failed";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: indexer workspace too small";
    case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT: a bounded device wait gave up";
    case CSA_ERR_DEVICE_CHECK: return "CSA_ERR_DEVICE_CHECK: a device bounds check failed";
    default: return "CSA: unknown status";
  }
}

int csa_version(void) { return 100; }

unsigned long long csa_kernel_launches(void) { return csa::g_launches.load(); }

csa_status_t csa_compress(const void* kv, long long kv_batch_stride, const void* score,
                          int score_width, void* out, long long out_batch_stride, int b, int sq,
                          int d, int ratio, csa_dtype_t dt, csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (kv == nullptr || score == nullptr || out == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(score) || !aligned16(out)) return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || d < 8 || d % 8 != 0 || ratio < 1 || sq < ratio)
    return CSA_ERR_INVALID_ARG;
  if (score_width != 1 && score_width != d) return CSA_ERR_INVALID_ARG;
  const int n_c = sq / ratio;
  if (kv_batch_stride < (long long)sq * d || out_batch_stride < (long long)n_c * d)
    return CSA_ERR_INVALID_ARG;
  const int esz = dt == CSA_BF16 ? 2 : 4;
  if ((kv_batch_stride * esz) % 16 != 0 || (out_batch_stride * esz) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (d > kMaxD) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_compress(kv, kv_batch_stride, score, score_width, out,
                                        out_batch_stride, b, sq, d, ratio, dt == CSA_BF16,
                                        (cudaStream_t)stream));
}

csa_status_t csa_compress_bwd(const void* kv, long long kv_batch_stride, const void* score,
                              int score_width, const float* dout, long long dout_batch_stride,
                              float* dkv, long long dkv_batch_stride, float* dscore, int b,
                              int sq, int d, int ratio, csa_dtype_t dt, csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (kv == nullptr || score == nullptr || dout == nullptr || dkv == nullptr || dscore == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(score) || !aligned16(dout) || !aligned16(dkv) ||
      !aligned16(dscore))
    return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || d < 8 || d % 8 != 0 || ratio < 1 || sq < ratio)
    return CSA_ERR_INVALID_ARG;
  if (score_width != 1 && score_width != d) return CSA_ERR_INVALID_ARG;
  const int n_c = sq / ratio;
  if (kv_batch_stride < (long long)sq * d || dkv_batch_stride < (long long)sq * d ||
      dout_batch_stride < (long long)n_c * d)
    return CSA_ERR_INVALID_ARG;
  const int esz = dt == CSA_BF16 ? 2 : 4;
  if ((kv_batch_stride * esz) % 16 != 0 || (dout_batch_stride * 4) % 16 != 0 ||
      (dkv_batch_stride * 4) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (d > kMaxD) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_compress_bwd(kv, kv_batch_stride, score, score_width, dout,
                                            dout_batch_stride, dkv, dkv_batch_stride, dscore, b,
                                            sq, d, ratio, dt == CSA_BF16, (cudaStream_t)stream));
}

csa_status_t csa_compress_overlap(const void* kv, long long kv_batch_stride, const void* score,
                                  int score_width, void* out, long long out_batch_stride, int b,
                                  int sq, int d, int ratio, int coff, csa_dtype_t dt,
                                  csa_stream_t stream) {
  if (coff < 1) return CSA_ERR_INVALID_ARG;
  if (coff == 1)
    return csa_compress(kv, kv_batch_stride, score, score_width, out, out_batch_stride, b, sq, d,
                        ratio, dt, stream);
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (kv == nullptr || score == nullptr || out == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(score) || !aligned16(out)) return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || d < 8 || d % 8 != 0 || ratio < 1 || sq < ratio)
    return CSA_ERR_INVALID_ARG;
  if (score_width != 1 && score_width != d) return CSA_ERR_INVALID_ARG;
  const int n_c = sq / ratio;
  if (kv_batch_stride < (long long)sq * d || out_batch_stride < (long long)n_c * d)
    return CSA_ERR_INVALID_ARG;
  const int esz = dt == CSA_BF16 ? 2 : 4;
  if ((kv_batch_stride * esz) % 16 != 0 || (out_batch_stride * esz) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (d > kMaxD || coff > 2) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_compress_overlap(kv, kv_batch_stride, score, score_width, out,
                                                out_batch_stride, b, sq, d, ratio, coff,
                                                dt == CSA_BF16, (cudaStream_t)stream));
}

csa_status_t csa_compress_overlap_bwd(const void* kv, long long kv_batch_stride,
                                      const void* score, int score_width, const float* dout,
                                      long long dout_batch_stride, float* dkv,
                                      long long dkv_batch_stride, float* dscore, int b, int sq,
                                      int d, int ratio, int coff, csa_dtype_t dt,
                                      csa_stream_t stream) {
  if (coff < 1) return CSA_ERR_INVALID_ARG;
  if (coff == 1)
    return csa_compress_bwd(kv, kv_batch_stride, score, score_width, dout, dout_batch_stride, dkv,
                            dkv_batch_stride, dscore, b, sq, d, ratio, dt, stream);
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (kv == nullptr || score == nullptr || dout == nullptr || dkv == nullptr || dscore == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(score) || !aligned16(dout) || !aligned16(dkv) ||
      !aligned16(dscore))
    return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || d < 8 || d % 8 != 0 || ratio < 1 || sq < ratio)
    return CSA_ERR_INVALID_ARG;
  if (score_width != 1 && score_width != d) return CSA_ERR_INVALID_ARG;
  const int n_c = sq / ratio;
  if (kv_batch_stride < (long long)sq * d || dkv_batch_stride < (long long)sq * d ||
      dout_batch_stride < (long long)n_c * d)
    return CSA_ERR_INVALID_ARG;
  const int esz = dt == CSA_BF16 ? 2 : 4;
  if ((kv_batch_stride * esz) % 16 != 0 || (dout_batch_stride * 4) % 16 != 0 ||
      (dkv_batch_stride * 4) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (d > kMaxD || coff > 2) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_compress_overlap_bwd(kv, kv_batch_stride, score, score_width, dout,
                                                    dout_batch_stride, dkv, dkv_batch_stride,
                                                    dscore, b, sq, d, ratio, coff,
                                                    dt == CSA_BF16, (cudaStream_t)stream));
}

// Arguments of the normalization and rotary embedding of the pooled rows.
static csa_status_t check_norm_rope(const float* weight, float eps, int rope_dim, float base,
                                    int d) {
  if (weight == nullptr || !aligned16(weight)) return CSA_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || eps > 1e30f) return CSA_ERR_INVALID_ARG;
  if (rope_dim < 0 || rope_dim > d || rope_dim % 2 != 0) return CSA_ERR_INVALID_ARG;
  if (rope_dim > 0 && !(base > 0.f && base < 1e30f)) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

csa_status_t csa_compress_norm_rope(const void* kv, long long kv_batch_stride, const void* score,
                                    int score_width, const float* norm_weight, float eps,
                                    int rope_dim, float rope_base, void* out,
                                    long long out_batch_stride, int b, int sq, int d, int ratio,
                                    csa_dtype_t dt, csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (kv == nullptr || score == nullptr || out == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(score) || !aligned16(out)) return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || d < 8 || d % 8 != 0 || ratio < 1 || sq < ratio)
    return CSA_ERR_INVALID_ARG;
  if (score_width != 1 && score_width != d) return CSA_ERR_INVALID_ARG;
  if (check_norm_rope(norm_weight, eps, rope_dim, rope_base, d) != CSA_OK)
    return CSA_ERR_INVALID_ARG;
  const int n_c = sq / ratio;
  if (kv_batch_stride < (long long)sq * d || out_batch_stride < (long long)n_c * d)
    return CSA_ERR_INVALID_ARG;
  const int esz = dt == CSA_BF16 ? 2 : 4;
  if ((kv_batch_stride * esz) % 16 != 0 || (out_batch_stride * esz) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (d > kMaxD) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_compress_norm_rope(kv, kv_batch_stride, score, score_width,
                                                  norm_weight, eps, rope_dim, rope_base, out,
                                                  out_batch_stride, b, sq, d, ratio,
                                                  dt == CSA_BF16, (cudaStream_t)stream));
}

csa_status_t csa_compress_norm_rope_bwd(const void* kv, long long kv_batch_stride,
                                        const void* score, int score_width,
                                        const float* norm_weight, float eps, int rope_dim,
                                        float rope_base, const float* dout,
                                        long long dout_batch_stride, float* dkv,
                                        long long dkv_batch_stride, float* dscore,
                                        float* dnorm_weight, int b, int sq, int d, int ratio,
                                        csa_dtype_t dt, csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (kv == nullptr || score == nullptr || dout == nullptr || dkv == nullptr ||
      dscore == nullptr || dnorm_weight == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(score) || !aligned16(dout) || !aligned16(dkv) ||
      !aligned16(dscore) || !aligned16(dnorm_weight))
    return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || d < 8 || d % 8 != 0 || ratio < 1 || sq < ratio)
    return CSA_ERR_INVALID_ARG;
  if (score_width != 1 && score_width != d) return CSA_ERR_INVALID_ARG;
  if (check_norm_rope(norm_weight, eps, rope_dim, rope_base, d) != CSA_OK)
    return CSA_ERR_INVALID_ARG;
  const int n_c = sq / ratio;
  if (kv_batch_stride < (long long)sq * d || dkv_batch_stride < (long long)sq * d ||
      dout_batch_stride < (long long)n_c * d)
    return CSA_ERR_INVALID_ARG;
  const int esz = dt == CSA_BF16 ? 2 : 4;
  if ((kv_batch_stride * esz) % 16 != 0 || (dout_batch_stride * 4) % 16 != 0 ||
      (dkv_batch_stride * 4) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (d > kMaxD) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_compress_norm_rope_bwd(
      kv, kv_batch_stride, score, score_width, norm_weight, eps, rope_dim, rope_base, dout,
      dout_batch_stride, dkv, dkv_batch_stride, dscore, dnorm_weight, b, sq, d, ratio,
      dt == CSA_BF16, (cudaStream_t)stream));
}

size_t csa_indexer_topk_min_workspace(int b, int n_c) {
  if (b < 1 || n_c < 1) return 0;
  return csa::indexer_min_chunk_bytes(b, n_c);
}

size_t csa_indexer_topk_workspace_size(int b, int sq, int n_c, int H_I, int d_I, int topk,
                                       csa_dtype_t dt) {
  (void)H_I; (void)d_I; (void)topk; (void)dt;
  if (b < 1 || sq < 1 || n_c < 1) return 0;
  const size_t full = (size_t)b * sq * n_c * sizeof(float);
  const size_t minimum = csa_indexer_topk_min_workspace(b, n_c);
  size_t ws = full < kDefaultIndexerWorkspace ? full : kDefaultIndexerWorkspace;
  if (ws < minimum) ws = minimum;
  return ws;
}

csa_status_t csa_indexer_topk_rows(const void* q_idx, const void* k_idx, const float* w,
                                   const int32_t* doc_ids, int32_t* topk_idx, float* topk_score,
                                   int b, int sq, int n_c, int H_I, int d_I, int ratio, int topk,
                                   csa_dtype_t dt, void* workspace, size_t workspace_bytes,
                                   int t_begin, int t_end, csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || k_idx == nullptr || w == nullptr || topk_idx == nullptr ||
      workspace == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(topk_idx) ||
      !aligned16(topk_score) || !aligned16(workspace) || !aligned16(doc_ids))
    return CSA_ERR_INVALID_ARG;
  const csa_status_t st = csa::check_indexer_shape(b, sq, n_c, H_I, d_I, ratio, topk, 8);
  if (st != CSA_OK) return st;
  if (check_rows(sq, t_begin, t_end) != CSA_OK) return CSA_ERR_INVALID_ARG;
  if (workspace_bytes < csa::indexer_min_chunk_bytes(b, n_c)) return CSA_ERR_WORKSPACE;
  const bool use_tc = dt == CSA_BF16 && !csa::indexer_cuda_cores_forced() &&
                      csa::indexer_tc_supported(H_I, d_I);
  int* status = device_status_ptr();
  cudaStream_t s = (cudaStream_t)stream;
  if (doc_ids != nullptr &&
      csa::launch_doc_boundary_check(doc_ids, b, sq, ratio, status, s) != cudaSuccess)
    return CSA_ERR_CUDA;
  return csa::indexer_chunks(b, sq, n_c, ratio, topk, doc_ids, topk_idx, topk_score, workspace,
                             workspace_bytes, s, t_begin, t_end, [&](float* ws, int t0, int nt) {
    return use_tc ? csa::launch_indexer_scores_tc(q_idx, k_idx, w, ws, t0, nt, b, sq, n_c, H_I,
                                                  d_I, ratio, status, s)
                  : csa::launch_indexer_scores_simt(q_idx, k_idx, w, ws, t0, nt, b, sq, n_c, H_I,
                                                    d_I, ratio, dt == CSA_BF16, s);
  });
}

csa_status_t csa_indexer_topk(const void* q_idx, const void* k_idx, const float* w,
                              const int32_t* doc_ids, int32_t* topk_idx, float* topk_score,
                              int b, int sq, int n_c, int H_I, int d_I, int ratio, int topk,
                              csa_dtype_t dt, void* workspace, size_t workspace_bytes,
                              csa_stream_t stream) {
  return csa_indexer_topk_rows(q_idx, k_idx, w, doc_ids, topk_idx, topk_score, b, sq, n_c, H_I,
                               d_I, ratio, topk, dt, workspace, workspace_bytes, 0, sq, stream);
}

csa_status_t csa_quantize_e4m3(const void* x, long long rows, int d, csa_dtype_t dt,
                               uint8_t* codes, float* scale, csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (rows < 0 || d < 8 || d % 8 != 0) return CSA_ERR_INVALID_ARG;
  if (rows == 0) return CSA_OK;
  if (x == nullptr || codes == nullptr || scale == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scale)) return CSA_ERR_INVALID_ARG;
  if (rows > (1ll << 33)) return CSA_ERR_UNSUPPORTED;   // grid of rows / 8 CTAs
  return from_cuda(csa::launch_quantize_e4m3(x, rows, d, dt == CSA_BF16, codes, scale,
                                             (cudaStream_t)stream));
}

csa_status_t csa_indexer_topk_fp8(const uint8_t* q8, const float* q_scale, const uint8_t* k8,
                                  const float* k_scale, const float* w, const int32_t* doc_ids,
                                  int32_t* topk_idx, float* topk_score, int b, int sq, int n_c,
                                  int H_I, int d_I, int ratio, int topk, void* workspace,
                                  size_t workspace_bytes, csa_stream_t stream) {
  if (q8 == nullptr || q_scale == nullptr || k8 == nullptr || k_scale == nullptr ||
      w == nullptr || topk_idx == nullptr || workspace == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(q_scale) || !aligned16(k8) || !aligned16(k_scale) ||
      !aligned16(w) || !aligned16(topk_idx) || !aligned16(topk_score) ||
      !aligned16(workspace) || !aligned16(doc_ids))
    return CSA_ERR_INVALID_ARG;
  const csa_status_t st = csa::check_indexer_shape(b, sq, n_c, H_I, d_I, ratio, topk, 16);
  if (st != CSA_OK) return st;
  if (workspace_bytes < csa::indexer_min_chunk_bytes(b, n_c)) return CSA_ERR_WORKSPACE;
  const bool use_tc = !csa::indexer_cuda_cores_forced() && csa::indexer_tc_fp8_supported(H_I, d_I);
  int* status = device_status_ptr();
  cudaStream_t s = (cudaStream_t)stream;
  if (doc_ids != nullptr &&
      csa::launch_doc_boundary_check(doc_ids, b, sq, ratio, status, s) != cudaSuccess)
    return CSA_ERR_CUDA;
  return csa::indexer_chunks(b, sq, n_c, ratio, topk, doc_ids, topk_idx, topk_score, workspace,
                             workspace_bytes, s, 0, sq, [&](float* ws, int t0, int nt) {
    return use_tc ? csa::launch_indexer_scores_tc(q8, k8, w, ws, t0, nt, b, sq, n_c, H_I, d_I,
                                                  ratio, status, s, q_scale, k_scale)
                  : csa::launch_indexer_scores_simt_fp8(q8, q_scale, k8, k_scale, w, ws, t0, nt,
                                                        b, sq, n_c, H_I, d_I, ratio, s);
  });
}

}  // extern "C"

namespace {

// CSA_ATTN_WARP_MMA=1 selects the warp-level mma.sync kernels for bf16 even
// where the tcgen05 kernels apply (the attention forward and backward, the
// indexer teacher and loss; same results up to rounding order).
bool warp_mma_forced() {
  const char* wm = getenv("CSA_ATTN_WARP_MMA");
  return wm != nullptr && wm[0] == '1';
}

csa_status_t attn_fwd_rows(const void* q, const void* kv_full, const int32_t* idx,
                           const float* sink, const int32_t* doc_ids, float scale, void* o,
                           float* lse, int b, int sq, int H, int d, int n_c, int ratio, int window,
                           int K, csa_dtype_t dt, int tb, int te, csa_stream_t stream) {
  csa_status_t st = check_attn(q, kv_full, idx, scale, b, sq, H, d, n_c, ratio, window, K, dt);
  if (st != CSA_OK) return st;
  if (check_rows(sq, tb, te) != CSA_OK) return CSA_ERR_INVALID_ARG;
  if (o == nullptr || lse == nullptr || !aligned16(o) || !aligned16(lse) || !aligned16(sink) ||
      !aligned16(doc_ids))
    return CSA_ERR_INVALID_ARG;
  const int Kl = idx ? K : n_c;
  cudaStream_t s = (cudaStream_t)stream;
  if (dt == CSA_BF16 && !warp_mma_forced() && csa::attn_tc_supported(H, d, n_c, Kl))
    return from_cuda(csa::launch_attn_fwd_tc(q, kv_full, idx, sink, scale, o, lse, b, sq, H, n_c,
                                             ratio, window, Kl, device_status_ptr(), s, doc_ids,
                                             tb, te));
  if (dt == CSA_BF16 && !warp_mma_forced() && csa::attn_tc512_supported(H, d, window, Kl))
    return from_cuda(csa::launch_attn_fwd_tc512(q, kv_full, idx, sink, scale, o, lse, b, sq,
                                                n_c, ratio, window, Kl, device_status_ptr(), s,
                                                doc_ids, tb, te));
  if (dt == CSA_BF16 && csa::attn_mma_supported(H, d, window, Kl))
    return from_cuda(csa::launch_attn_fwd_mma(q, kv_full, idx, sink, scale, o, lse, b, sq, H, d,
                                              n_c, ratio, window, Kl, s, doc_ids, tb, te));
  return from_cuda(csa::launch_attn_fwd_simt(q, kv_full, idx, sink, scale, o, lse, b, sq, H, d,
                                             n_c, ratio, window, Kl, dt == CSA_BF16, s, doc_ids,
                                             tb, te));
}

csa_status_t attn_bwd_rows(const void* q, const void* kv_full, const int32_t* idx,
                           const float* sink, const int32_t* doc_ids, float scale, const void* o,
                           const float* lse, const void* dO, float* dq, float* dkv, float* dsink,
                           int b, int sq, int H, int d, int n_c, int ratio, int window, int K,
                           csa_dtype_t dt, int tb, int te, bool accumulate, csa_stream_t stream) {
  csa_status_t st = check_attn(q, kv_full, idx, scale, b, sq, H, d, n_c, ratio, window, K, dt);
  if (st != CSA_OK) return st;
  if (check_rows(sq, tb, te) != CSA_OK) return CSA_ERR_INVALID_ARG;
  if (o == nullptr || lse == nullptr || dO == nullptr || dq == nullptr || dkv == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (sink != nullptr && dsink == nullptr) return CSA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(lse) || !aligned16(dO) || !aligned16(dq) || !aligned16(dkv) ||
      !aligned16(dsink) || !aligned16(sink) || !aligned16(doc_ids))
    return CSA_ERR_INVALID_ARG;
  const int Kl = idx ? K : n_c;
  cudaStream_t s = (cudaStream_t)stream;
  const int n_kv = sq + n_c;
  if (!accumulate) {
    cudaError_t e = csa::launch_zero_f32_pair(dkv, (size_t)b * n_kv * d, dsink,
                                              dsink != nullptr ? (size_t)H : 0, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  }
  if (dt == CSA_BF16 && !warp_mma_forced() && csa::attn_tc_bwd_supported(H, d, n_c, Kl))
    return from_cuda(csa::launch_attn_bwd_tc(q, kv_full, idx, sink, scale, o, lse, dO, dq, dkv,
                                             dsink, b, sq, H, n_c, ratio, window, Kl,
                                             device_status_ptr(), s, doc_ids, tb, te));
  if (dt == CSA_BF16 && !warp_mma_forced() && csa::attn_tc512_bwd_supported(H, d, window, Kl))
    return from_cuda(csa::launch_attn_bwd_tc512(q, kv_full, idx, sink, scale, lse, dO, dq, dkv,
                                                dsink, b, sq, n_c, ratio, window, Kl,
                                                device_status_ptr(), s, doc_ids, tb, te));
  if (dt == CSA_BF16 && csa::attn_mma_supported(H, d, window, Kl))
    return from_cuda(csa::launch_attn_bwd_mma(q, kv_full, idx, sink, scale, o, lse, dO, dq, dkv,
                                              dsink, b, sq, H, d, n_c, ratio, window, Kl, s,
                                              doc_ids, tb, te));
  return from_cuda(csa::launch_attn_bwd_simt(q, kv_full, idx, sink, scale, o, lse, dO, dq, dkv,
                                             dsink, b, sq, H, d, n_c, ratio, window, Kl,
                                             dt == CSA_BF16, s, doc_ids, tb, te));
}

}  // namespace

extern "C" {

csa_status_t csa_attn_fwd(const void* q, const void* kv_full, const int32_t* idx,
                          const float* sink, const int32_t* doc_ids, float scale, void* o,
                          float* lse, int b, int sq, int H, int d, int n_c, int ratio, int window,
                          int K, csa_dtype_t dt, csa_stream_t stream) {
  return attn_fwd_rows(q, kv_full, idx, sink, doc_ids, scale, o, lse, b, sq, H, d, n_c, ratio,
                       window, K, dt, 0, sq, stream);
}

csa_status_t csa_attn_bwd(const void* q, const void* kv_full, const int32_t* idx,
                          const float* sink, const int32_t* doc_ids, float scale, const void* o,
                          const float* lse, const void* dO, float* dq, float* dkv, float* dsink,
                          int b, int sq, int H, int d, int n_c, int ratio, int window, int K,
                          csa_dtype_t dt, csa_stream_t stream) {
  return attn_bwd_rows(q, kv_full, idx, sink, doc_ids, scale, o, lse, dO, dq, dkv, dsink, b, sq,
                       H, d, n_c, ratio, window, K, dt, 0, sq, false, stream);
}

csa_status_t csa_attn_fwd_rows(const void* q, const void* kv_full, const int32_t* idx,
                               const float* sink, const int32_t* doc_ids, float scale, void* o,
                               float* lse, int b, int sq, int H, int d, int n_c, int ratio,
                               int window, int K, csa_dtype_t dt, int t_begin, int t_end,
                               csa_stream_t stream) {
  return attn_fwd_rows(q, kv_full, idx, sink, doc_ids, scale, o, lse, b, sq, H, d, n_c, ratio,
                       window, K, dt, t_begin, t_end, stream);
}

csa_status_t csa_attn_bwd_rows(const void* q, const void* kv_full, const int32_t* idx,
                               const float* sink, const int32_t* doc_ids, float scale,
                               const void* o, const float* lse, const void* dO, float* dq,
                               float* dkv, float* dsink, int b, int sq, int H, int d, int n_c,
                               int ratio, int window, int K, csa_dtype_t dt, int t_begin,
                               int t_end, int accumulate, csa_stream_t stream) {
  return attn_bwd_rows(q, kv_full, idx, sink, doc_ids, scale, o, lse, dO, dq, dkv, dsink, b, sq,
                       H, d, n_c, ratio, window, K, dt, t_begin, t_end, accumulate != 0, stream);
}

csa_status_t csa_indexer_teacher(const void* q, const void* kv_full, const int32_t* idx,
                                 const float* lse, float scale, float* target, int b, int sq,
                                 int H, int d, int n_c, int ratio, int K, csa_dtype_t dt,
                                 csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (q == nullptr || kv_full == nullptr || idx == nullptr || lse == nullptr ||
      target == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_full) || !aligned16(idx) || !aligned16(lse) ||
      !aligned16(target))
    return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || H < 1 || d < 8 || d % 8 != 0 || ratio < 1 || K < 1)
    return CSA_ERR_INVALID_ARG;
  if (sq < ratio || n_c != sq / ratio || !(scale == scale)) return CSA_ERR_INVALID_ARG;
  if (d > kMaxD || H > kMaxH || n_c > kMaxNc) return CSA_ERR_UNSUPPORTED;
  if (dt == CSA_BF16 && !warp_mma_forced() && csa::indexer_teacher_tc_supported(H, d, n_c, K))
    return from_cuda(csa::launch_indexer_teacher_tc(q, kv_full, idx, lse, scale, target, b, sq, H,
                                                    n_c, ratio, K, device_status_ptr(),
                                                    (cudaStream_t)stream));
  const bool mma = dt == CSA_BF16 && csa::indexer_teacher_mma_ok(H, d);
  if (csa::indexer_teacher_smem(mma, H, d, K) > 227 * 1024) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_indexer_teacher(q, kv_full, idx, lse, scale, target, b, sq, H, d,
                                               n_c, ratio, K, dt == CSA_BF16,
                                               (cudaStream_t)stream));
}

csa_status_t csa_indexer_loss(const void* q_idx, const void* k_idx, const float* w,
                              const int32_t* idx, const float* target, float* loss,
                              float* dq_idx, float* dk_idx, float* dw, int b, int sq, int n_c,
                              int H_I, int d_I, int ratio, int K, csa_dtype_t dt,
                              csa_stream_t stream) {
  if (!valid_dtype(dt)) return CSA_ERR_INVALID_ARG;
  if (q_idx == nullptr || k_idx == nullptr || w == nullptr || idx == nullptr ||
      target == nullptr || loss == nullptr || dq_idx == nullptr || dk_idx == nullptr ||
      dw == nullptr)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(idx) ||
      !aligned16(target) || !aligned16(loss) || !aligned16(dq_idx) || !aligned16(dk_idx) ||
      !aligned16(dw))
    return CSA_ERR_INVALID_ARG;
  if (b < 1 || sq < 1 || H_I < 1 || d_I < 8 || d_I % 8 != 0 || ratio < 1 || K < 1)
    return CSA_ERR_INVALID_ARG;
  if (sq < ratio || n_c != sq / ratio) return CSA_ERR_INVALID_ARG;
  if (d_I > kMaxDI || H_I > kMaxH || n_c > kMaxNc) return CSA_ERR_UNSUPPORTED;
  if (dt == CSA_BF16 && !warp_mma_forced() && csa::indexer_loss_tc_supported(H_I, d_I, n_c)) {
    int* status = device_status_ptr();
    if (status == nullptr) return CSA_ERR_CUDA;
    return from_cuda(csa::launch_indexer_loss_tc(q_idx, k_idx, w, idx, target, loss, dq_idx,
                                                 dk_idx, dw, b, sq, H_I, n_c, ratio, K, status,
                                                 (cudaStream_t)stream));
  }
  const bool mma = dt == CSA_BF16 && csa::indexer_loss_mma_ok(H_I, d_I);
  if (csa::indexer_loss_smem(mma, H_I, d_I, K) > 227 * 1024) return CSA_ERR_UNSUPPORTED;
  return from_cuda(csa::launch_indexer_loss(q_idx, k_idx, w, idx, target, loss, dq_idx, dk_idx,
                                            dw, b, sq, H_I, d_I, n_c, ratio, K, dt == CSA_BF16,
                                            (cudaStream_t)stream));
}

csa_status_t csa_debug_arm_fault(int site) {
  if (site < 0) return CSA_ERR_INVALID_ARG;
  int* p = device_status_ptr();
  if (p == nullptr) return CSA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return CSA_ERR_CUDA;
  return from_cuda(cudaMemcpy(p + 2, &site, sizeof(int), cudaMemcpyHostToDevice));
}

csa_status_t csa_get_device_status(csa_stream_t stream, int* status_out, int* site_out) {
  if (status_out == nullptr) return CSA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CSA_ERR_CUDA;
  int* p = device_status_ptr();
  if (p == nullptr) return CSA_ERR_CUDA;
  int v[2] = {0, 0};
  if (cudaMemcpy(v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  const int zero[2] = {0, 0};
  if (cudaMemcpy(p, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return CSA_ERR_CUDA;
  *status_out = v[0];
  if (site_out != nullptr) *site_out = v[1];
  return CSA_OK;
}

}  // extern "C"
