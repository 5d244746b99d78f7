// Host-side launchers of the CSA kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace csa {

// Compressor: softmax-weighted pooling.
cudaError_t launch_compress(const void* kv, long long kv_bs, const void* score, int score_width,
                            void* out, long long out_bs, int b, int sq, int d, int ratio,
                            bool bf16, cudaStream_t s);

// Exact per-row top-K of the chunk of scores in ws (rows [t0, t0+nt) of every
// batch element, laid out [b][nt][n_c]).  doc (nullable, [b][sq]): per-token
// document ids; a block is a candidate only for queries of its document.
cudaError_t launch_topk_select(const float* ws, int32_t* topk_idx, float* topk_score, int t0,
                               int nt, int b, int sq, int n_c, int ratio, int K, cudaStream_t s,
                               const int32_t* doc = nullptr);

// Record CSA_ERR_DEVICE_CHECK when a packed document starts inside a
// compressed block (doc [b][sq]).
cudaError_t launch_doc_boundary_check(const int32_t* doc, int b, int sq, int ratio, int* status,
                                      cudaStream_t s);

cudaError_t launch_compress_bwd(const void* kv, long long kv_bs, const void* score,
                                int score_width, const float* g, long long g_bs, float* dkv,
                                long long dkv_bs, float* dscore, int b, int sq, int d, int ratio,
                                bool bf16, cudaStream_t s);

// Overlapping compression (coff blocks per pooling window; coff 1 = the above).
cudaError_t launch_compress_overlap(const void* kv, long long kv_bs, const void* score,
                                    int score_width, void* out, long long out_bs, int b, int sq,
                                    int d, int ratio, int coff, bool bf16, cudaStream_t s);
cudaError_t launch_compress_overlap_bwd(const void* kv, long long kv_bs, const void* score,
                                        int score_width, const float* g, long long g_bs,
                                        float* dkv, long long dkv_bs, float* dscore, int b,
                                        int sq, int d, int ratio, int coff, bool bf16,
                                        cudaStream_t s);

// Compressor followed by the RMS normalization and the rotary embedding of
// each pooled row, and the gradient of the three (dweight [d] zeroed here).
cudaError_t launch_compress_norm_rope(const void* kv, long long kv_bs, const void* score,
                                      int score_width, const float* weight, float eps,
                                      int rope_dim, float base, void* out, long long out_bs,
                                      int b, int sq, int d, int ratio, bool bf16, cudaStream_t s);
cudaError_t launch_compress_norm_rope_bwd(const void* kv, long long kv_bs, const void* score,
                                          int score_width, const float* weight, float eps,
                                          int rope_dim, float base, const float* g,
                                          long long g_bs, float* dkv, long long dkv_bs,
                                          float* dscore, float* dweight, int b, int sq, int d,
                                          int ratio, bool bf16, cudaStream_t s);

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t s);
// Two buffers in one launch (b may be null with nb = 0).
cudaError_t launch_zero_f32_pair(float* a, size_t na, float* b, size_t nb, cudaStream_t s);

}  // namespace csa
