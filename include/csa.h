/*
 * csa.h - C ABI of the Compressed Sparse Attention (CSA) hot path.
 *
 * One CSA layer on one GPU, as four calls (plus helpers):
 *
 *   csa_compress      softmax-weighted pooling of `ratio` consecutive KV tokens
 *                     (csa_compress_bwd: its gradient)
 *   csa_indexer_topk  lightning-indexer scores fused with an exact causal top-k
 *   csa_attn_fwd      sparse MQA (shared K=V) over window + top-k compressed
 *                     rows + per-head sink; returns O and LSE
 *   csa_attn_bwd      dQ, dKV, dSink, accumulated in fp32
 *
 * Further calls: the normalization and rotary embedding of the pooled rows
 * (csa_compress_norm_rope and its backward), packed documents (the doc_ids
 * argument of the indexer and the attention), the indexer's training path
 * (csa_indexer_teacher,
 * csa_indexer_loss), overlapping compression (csa_compress_overlap and its
 * backward), an FP8 indexer (csa_quantize_e4m3, csa_indexer_topk_fp8), an
 * indexer that needs no caller workspace (csa_indexer_topk_noalloc) and
 * row-range forms of the indexer and the attention for a layer split by
 * query rows across GPUs (csa_*_rows).
 *
 * Sources (page title, section):
 *   "Add unfused SBHD compressed sparse attention" (Megatron-LM PR #6400):
 *     compressor review, causal compressed mask, indexer / top-k block,
 *     review of the gather backward, attention-sink parameter.
 *   "Refactor Deepseek v4 to use Attention Gym's Compressed Sparse Attention"
 *     (torchtitan PR #4452): the selected_attention operator (window +
 *     selected compressed entries + sink in one softmax, per-head LSE).
 *   "Add the min-memory DSA attention kernels" (Megatron-LM PR #7152):
 *     streamed score tiles, tie-exact top-k, fp32 scatter of repeated keys.
 *
 * Notation: b batch, sq query tokens, H query heads, d shared K=V head dim,
 * r = ratio, n_c = sq / r (integer division), n_kv = sq + n_c,
 * vis(t) = (t + 1) / r (integer division), W = window,
 * K = min(topk, n_c), H_I / d_I = indexer heads / head dim.
 *
 * Layouts (all row-major, innermost dimension contiguous, batch-major):
 *   kv_full  [b, n_kv, d]   raw rows 0..sq-1, then compressed rows sq..n_kv-1
 *   q, o, dO [b, sq, H, d]
 *   lse      [b, sq, H]     fp32, natural log, sink included
 *   idx      [b, sq, K]     int32, compressed-relative block ids, -1 = pad
 *   sink     [H]            fp32 logits (NULL = no sink = -inf)
 *   q_idx    [b, sq, H_I, d_I], k_idx [b, n_c, d_I], w [b, sq, H_I] fp32
 *
 * Ownership: the caller allocates and owns every buffer (including the
 * indexer workspace).  The library keeps no per-call state and allocates
 * no memory.  All pointers except `workspace` sizes are device pointers.
 *
 * Execution: every call only validates its arguments on the host and
 * enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  No call synchronizes.  Argument errors are detected before any
 * CUDA call, so an invalid call has no effect on the device.
 *
 * Errors: the return value covers host-side validation and launch errors.
 * Conditions found on the device (a bounded wait that gave up, a device
 * check that failed) are recorded in a per-device status word, read and
 * cleared by csa_get_device_status().
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or shape */
  CSA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype, d > 512, ...) */
  CSA_ERR_CUDA = 3,         /* a CUDA launch or runtime call failed */
  CSA_ERR_WORKSPACE = 4,    /* indexer workspace too small */
  CSA_ERR_TIMEOUT = 5,      /* device: a bounded wait gave up */
  CSA_ERR_DEVICE_CHECK = 6  /* device: a consistency or input check failed */
} csa_status_t;

typedef enum { CSA_FP32 = 0, CSA_BF16 = 1 } csa_dtype_t;

typedef void* csa_stream_t; /* cudaStream_t */

/* Static, never-freed description of a status code. */
const char* csa_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int csa_version(void);

/* Number of kernels this library has enqueued in this process (all
 * devices, all calls): lets a caller count the launches of a timed region. */
unsigned long long csa_kernel_launches(void);

/*
 * csa_compress - softmax-weighted pooling of ratio consecutive tokens.
 *
 * Defined by the compressor review of "Add unfused SBHD compressed sparse
 * attention": for block j < n_c and channel c,
 *   weights_t = softmax over t in [j*r, (j+1)*r) of score[b, t, c'],
 *   out[b, j, c] = sum_t weights_t * kv[b, t, c],
 * with c' = c when score_width == d and c' = 0 when score_width == 1.
 * The softmax, products and sum run in fp32; the result is cast once to dt.
 * Tokens past the last complete block (sq % r of them) are not pooled.
 *
 *   kv      in   [b, sq, d] rows of dt; batch stride kv_batch_stride elements
 *                (sq*d for a packed tensor, n_kv*d when kv lives in kv_full)
 *   score   in   [b, sq, score_width] of dt, packed
 *   out     out  [b, n_c, d] rows of dt; batch stride out_batch_stride
 *                elements (pass kv_full + sq*d and n_kv*d to write the
 *                compressed rows of kv_full in place)
 * Errors: INVALID_ARG for null pointers, pointers not 16-byte aligned,
 * d % 8 != 0, score_width not in {1, d}, ratio < 1, sq < ratio, strides
 * smaller than a batch's rows; UNSUPPORTED for d > 512.
 */
csa_status_t csa_compress(const void* kv, long long kv_batch_stride,
                          const void* score, int score_width,
                          void* out, long long out_batch_stride,
                          int b, int sq, int d, int ratio,
                          csa_dtype_t dt, csa_stream_t stream);

/*
 * csa_compress_bwd - gradient of csa_compress.
 *
 * With w_t the softmax weights of block j and channel c (as in csa_compress)
 * and g = dout[b, j, c] the gradient of the pooled row:
 *   dkv[b, t, c]    += w_t * g                         (accumulated)
 *   dscore[b, t, c'] = w_t * g * (kv[b, t, c] - out[b, j, c])
 * summed over c for score_width == 1 (c' = 0).  The pooled row is recomputed
 * in fp32.  Tokens past the last complete block: dkv unchanged, dscore 0.
 * dkv accumulates so that the raw rows of the attention's dkv
 * (dkv_full[:, :sq]) receive the compressor's share in place.
 *
 *   kv, score  in   as csa_compress
 *   dout       in   [b, n_c, d] fp32, batch stride dout_batch_stride (pass
 *                   dkv_full + sq*d and n_kv*d for the compressed rows)
 *   dkv        in/out [b, sq, d] fp32, batch stride dkv_batch_stride
 *   dscore     out  [b, sq, score_width] fp32, packed, fully written
 * Errors: as csa_compress (all pointers 16-byte aligned, strides in elements).
 * The pages keep this pooling in fp32 and cast once ("Add unfused SBHD
 * compressed sparse attention", compressor review, which also describes the
 * test of the KV and score gradients against an fp32 pooling oracle).
 */
csa_status_t csa_compress_bwd(const void* kv, long long kv_batch_stride,
                              const void* score, int score_width,
                              const float* dout, long long dout_batch_stride,
                              float* dkv, long long dkv_batch_stride, float* dscore,
                              int b, int sq, int d, int ratio,
                              csa_dtype_t dt, csa_stream_t stream);

/*
 * csa_compress_overlap - csa_compress with overlapping pooling windows.
 *
 * The compressor review of "Add unfused SBHD compressed sparse attention"
 * calls ratio 128 "non-overlapping, coff = 1"; this call takes coff, the
 * number of ratio-blocks each compressed entry pools (the library's reading:
 * the window ends with the entry's own block).  For entry j < n_c:
 *   window(j) = tokens [max(0, (j + 1 - coff) * r), (j + 1) * r)
 *   weights_t = softmax over t in window(j) of score[b, t, c'],
 *   out[b, j, c] = sum_t weights_t * kv[b, t, c]
 * in fp32, cast once.  coff = 1 is csa_compress; the first coff - 1 entries
 * pool the tokens that exist.  Arguments as csa_compress.
 * Errors: as csa_compress; INVALID_ARG for coff < 1, UNSUPPORTED for coff > 2.
 */
csa_status_t csa_compress_overlap(const void* kv, long long kv_batch_stride,
                                  const void* score, int score_width,
                                  void* out, long long out_batch_stride,
                                  int b, int sq, int d, int ratio, int coff,
                                  csa_dtype_t dt, csa_stream_t stream);

/*
 * csa_compress_overlap_bwd - gradient of csa_compress_overlap.
 *
 * Each entry j contributes, for t in window(j), with its weights w_t and
 * g = dout[b, j, c]:
 *   dkv[b, t, c]     += w_t * g
 *   dscore[b, t, c'] += w_t * g * (kv[b, t, c] - out[b, j, c])
 * so a token in several windows sums their contributions (dkv accumulates
 * into what it holds; dscore is fully written).  Arguments and errors as
 * csa_compress_bwd, plus coff as in csa_compress_overlap.
 */
csa_status_t csa_compress_overlap_bwd(const void* kv, long long kv_batch_stride,
                                      const void* score, int score_width,
                                      const float* dout, long long dout_batch_stride,
                                      float* dkv, long long dkv_batch_stride, float* dscore,
                                      int b, int sq, int d, int ratio, int coff,
                                      csa_dtype_t dt, csa_stream_t stream);

/*
 * csa_compress_norm_rope - csa_compress followed by the normalization and the
 * rotary embedding of each pooled row.
 *
 * "Add unfused SBHD compressed sparse attention", compressor review: the
 * pooled row is cast once to dt and then normalized (kv = self.norm(kv));
 * its config fields give the rotary base of compressed KV positions
 * (csa_compress_rotary_base = 40000).  The norm's type, the rotary channels
 * and the compressed positions are not given; this call's readings: with x
 * the pooled row after its cast to dt,
 *   y = x / sqrt(mean_c(x^2) + eps) * norm_weight          (fp32)
 *   y[2i'], y[2i'+1] of the last rope_dim channels (i' = the pair's index in
 *   the rotary part, channel pairs interleaved) turned by the angle
 *   pos_j * rope_base^(-2 i' / rope_dim), pos_j = (j+1)*ratio - 1 (the
 *   position of the entry's last pooled token),
 *   out[b, j, :] = y cast once to dt.
 * The angles are formed in double precision.  rope_dim = 0: no rotation.
 *
 *   kv, score, out, strides, sizes, dt   as csa_compress
 *   norm_weight  in  [d] fp32, 16-byte aligned
 *   eps          >= 0 (finite)
 *   rope_dim     even, 0 <= rope_dim <= d;  rope_base > 0 when rope_dim > 0
 * Errors: as csa_compress, plus INVALID_ARG for a null or misaligned weight,
 * a negative or non-finite eps, an odd or out-of-range rope_dim, a
 * non-positive rope_base.
 */
csa_status_t csa_compress_norm_rope(const void* kv, long long kv_batch_stride,
                                    const void* score, int score_width,
                                    const float* norm_weight, float eps, int rope_dim,
                                    float rope_base, void* out, long long out_batch_stride,
                                    int b, int sq, int d, int ratio, csa_dtype_t dt,
                                    csa_stream_t stream);

/*
 * csa_compress_norm_rope_bwd - gradient of csa_compress_norm_rope.
 *
 * dout [b, n_c, d] fp32 (batch stride dout_batch_stride) is the gradient of
 * the output rows.  With x the cast pooled row, xh = x / rms and dy = dout
 * turned back by the rotation's angle:
 *   dnorm_weight[c] = sum over all rows of dy[c] * xh[c]  (zeroed by the call)
 *   dx = (dy * norm_weight - xh * mean_c(dy * norm_weight * xh)) / rms
 * and dx passes the cast unchanged into the pooling's gradient, as in
 * csa_compress_bwd: dkv += w_t dx (accumulated), dscore written.
 *   other arguments as csa_compress_bwd and csa_compress_norm_rope
 * Errors: as csa_compress_bwd, plus those of csa_compress_norm_rope and
 * INVALID_ARG for a null dnorm_weight.  dnorm_weight is summed with fp32
 * atomics (reproducible to rounding only).
 */
csa_status_t csa_compress_norm_rope_bwd(const void* kv, long long kv_batch_stride,
                                        const void* score, int score_width,
                                        const float* norm_weight, float eps, int rope_dim,
                                        float rope_base, const float* dout,
                                        long long dout_batch_stride, float* dkv,
                                        long long dkv_batch_stride, float* dscore,
                                        float* dnorm_weight, int b, int sq, int d, int ratio,
                                        csa_dtype_t dt, csa_stream_t stream);

/*
 * Bytes of indexer workspace that csa_indexer_topk uses by default: the
 * fp32 score rows of one chunk of queries (n_c floats per query row, at
 * most 128 MiB, at least one 128-row tile).  Any workspace of at least
 * csa_indexer_topk_min_workspace() bytes works: the call then processes
 * the b*sq query rows in chunks that fit, so peak memory follows the
 * workspace, not sq * n_c.  Returns 0 for invalid sizes.
 */
size_t csa_indexer_topk_workspace_size(int b, int sq, int n_c, int H_I, int d_I,
                                       int topk, csa_dtype_t dt);
size_t csa_indexer_topk_min_workspace(int b, int n_c);

/*
 * csa_indexer_topk - lightning indexer + causal top-k.
 *
 * Scores ("Add unfused SBHD compressed sparse attention", indexer block;
 * "Refactor Deepseek v4 ...", indexer selectability):
 *   I[b,t,j] = sum_h w[b,t,h] * max(0, q_idx[b,t,h,:] . k_idx[b,j,:]),
 *   for the visible blocks j < vis(t).  w is used as given (the caller
 *   folds any softmax scale into it).
 * Selection ("Add the min-memory DSA attention kernels": tie-exact routing,
 * support sorted by position): the K = min(topk, n_c) largest scores of the
 * row, ties to the lower j, written in ascending j; rows with fewer than K
 * candidates hold all of them followed by -1.
 * Packed documents ("Refactor Deepseek v4 ...", doc_ids isolation): with
 * doc_ids, block j covers tokens [j*ratio, (j+1)*ratio), belongs to
 * doc_ids[b, j*ratio], and is a candidate for query t only when
 * doc_ids[b,t] == doc_ids[b, j*ratio] (and j < vis(t)).  Documents are
 * expected to start on multiples of ratio, so that no block mixes two.
 * Products are bf16 x bf16 (or fp32 x fp32) with fp32 accumulation; the
 * selection compares the fp32 scores exactly (-0 equals +0).
 *
 *   q_idx       in   [b, sq, H_I, d_I] dt
 *   k_idx       in   [b, n_c, d_I]     dt
 *   w           in   [b, sq, H_I]      fp32
 *   doc_ids     in   [b, sq]           int32 document id per token; NULL =
 *                                      one document (every visible block)
 *   topk_idx    out  [b, sq, K]        int32
 *   topk_score  out  [b, sq, K]        fp32 scores of the selected blocks
 *                                      (0 at -1 slots); may be NULL
 *   workspace   scratch, device, 16-byte aligned, >= min workspace
 * Errors: INVALID_ARG (null or misaligned pointers, d_I % 8 != 0,
 * n_c != sq / ratio, topk < 1, H_I < 1); WORKSPACE (too small);
 * UNSUPPORTED (d_I > 256, n_c > 16384).
 */
csa_status_t csa_indexer_topk(const void* q_idx, const void* k_idx, const float* w,
                              const int32_t* doc_ids, int32_t* topk_idx, float* topk_score,
                              int b, int sq, int n_c, int H_I, int d_I, int ratio, int topk,
                              csa_dtype_t dt, void* workspace, size_t workspace_bytes,
                              csa_stream_t stream);

/*
 * csa_quantize_e4m3 - per-row e4m3 quantization, the input format of
 * csa_indexer_topk_fp8.
 *
 * The pages name indexer quantization among the parts not yet included
 * ("Refactor Deepseek v4 ...", the V4.1-Flash backbone's list of what is
 * not included); this per-row rule is the library's own reading.  For each
 * row r of x (the last axis, d elements):
 *   amax     = max_c |x[r,c]|                     (fp32)
 *   scale[r] = amax / 448                          (fp32, rounded once)
 *   codes[r,c] = e4m3(x[r,c] * (448 / amax))       (fp32 reciprocal and
 *                product, each rounded to nearest; then to nearest-even
 *                e4m3, saturating at +-448; no NaN codes)
 * An all-zero row gets scale 0 and zero codes.  Every step is a correctly
 * rounded fp32 operation, so the result is reproducible bit for bit.
 *
 *   x      in   [rows, d] dt (bf16 or fp32), 16-byte aligned
 *   codes  out  [rows, d] uint8 e4m3 bit patterns (OCP FP8 E4M3FN)
 *   scale  out  [rows]    fp32
 * For csa_indexer_topk_fp8, q_idx [b, sq, H_I, d_I] is quantized as
 * rows = b*sq*H_I and k_idx [b, n_c, d_I] as rows = b*n_c.
 * Errors: INVALID_ARG (null or misaligned pointers, d % 8 != 0, d < 8,
 * rows < 0); UNSUPPORTED (rows > 2^33).  rows == 0 is a no-op.
 */
csa_status_t csa_quantize_e4m3(const void* x, long long rows, int d, csa_dtype_t dt,
                               uint8_t* codes, float* scale, csa_stream_t stream);

/*
 * csa_indexer_topk_fp8 - csa_indexer_topk on e4m3 codes with per-row scales.
 *
 * Scores, with the codes' exact values q8, k8 and the scales q_scale,
 * k_scale of csa_quantize_e4m3 (non-negative, so they commute with the ReLU):
 *   I[b,t,j] = k_scale[b,j] * sum_h (w[b,t,h] * q_scale[b,t,h])
 *                                   * max(0, q8[b,t,h,:] . k8[b,j,:])
 * for the visible (and, with doc_ids, same-document) blocks; the selection,
 * the output layout, doc_ids and the workspace rules are those of
 * csa_indexer_topk.  The code products are exact in the fp32 accumulators
 * (tcgen05 kind::f8f6f4 for d_I in {128, 256} and H_I <= 64, a CUDA-core
 * kernel otherwise).
 *
 *   q8       in  [b, sq, H_I, d_I] uint8 e4m3 codes
 *   q_scale  in  [b, sq, H_I]      fp32
 *   k8       in  [b, n_c, d_I]     uint8 e4m3 codes
 *   k_scale  in  [b, n_c]          fp32
 *   other arguments as csa_indexer_topk
 * Errors: as csa_indexer_topk, with d_I % 16 != 0 (instead of % 8) and a
 * null scale pointer also INVALID_ARG.
 */
csa_status_t csa_indexer_topk_fp8(const uint8_t* q8, const float* q_scale, const uint8_t* k8,
                                  const float* k_scale, const float* w, const int32_t* doc_ids,
                                  int32_t* topk_idx, float* topk_score, int b, int sq, int n_c,
                                  int H_I, int d_I, int ratio, int topk, void* workspace,
                                  size_t workspace_bytes, csa_stream_t stream);

/*
 * csa_indexer_topk_noalloc - csa_indexer_topk for callers that cannot
 * allocate device memory.
 *
 * The pages have no counterpart to this call.  csa_indexer_topk needs a
 * scratch workspace from its caller; some callers cannot provide one: a
 * plugin or custom operator inside a framework that owns all device memory
 * and gives it no allocator, a serving loop that must not call cudaMalloc
 * once it runs (cudaMalloc may synchronize the whole device), a C caller
 * with no spare buffer.  This call takes the arguments of csa_indexer_topk
 * minus the workspace and minus doc_ids, and returns the results that
 * csa_indexer_topk returns with doc_ids == NULL: every batch row is one
 * document (packed-document callers use csa_indexer_topk).  The score rows it
 * needs live in a fixed array of CSA_NOALLOC_SCRATCH_BYTES in the library's
 * own device memory.
 *
 *  - Memory: every GPU that loads the library holds the array until the
 *    process exits.  The call allocates nothing (no cudaMalloc, no cudaFree,
 *    no allocating library routine).
 *  - Limit: the query rows are processed in chunks that fit the array; a
 *    problem whose smallest chunk does not fit (b * 128 * n_c * 4 bytes >
 *    CSA_NOALLOC_SCRATCH_BYTES) is rejected with CSA_ERR_WORKSPACE before any
 *    work is enqueued.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress, no allocation) with that device current;
 *    make that first call before any stream capture.  The address is kept
 *    for the life of the process and is not looked up again after a
 *    cudaDeviceReset of that device: do not call this entry point on a
 *    device after resetting it.
 *  - Sharing: all calls on a device use the same array, which keeps the last
 *    call's scores.  Every value a call reads is written earlier in the same
 *    call, so nothing needs clearing, but two calls whose work overlaps on the
 *    GPU (different streams, or different host threads on one device) race
 *    and corrupt each other's results: order them on one stream or with
 *    events.
 * Errors: as csa_indexer_topk, with CSA_ERR_WORKSPACE for the limit above.
 */
#define CSA_NOALLOC_SCRATCH_BYTES (16u << 20)
csa_status_t csa_indexer_topk_noalloc(const void* q_idx, const void* k_idx, const float* w,
                                      int32_t* topk_idx, float* topk_score,
                                      int b, int sq, int n_c, int H_I, int d_I, int ratio,
                                      int topk, csa_dtype_t dt, csa_stream_t stream);

/*
 * csa_attn_fwd - sparse MQA forward with sink.
 *
 * Defined by "Add unfused SBHD compressed sparse attention" (unfused sparse
 * core: gather of the selected rows of the compact KV buffer, the two
 * einsums, the invalid mask; sink parameter; softmax_scale) and by the
 * selected_attention operator of "Refactor Deepseek v4 ..." (window +
 * selected compressed entries + sink in one softmax, returns LSE).
 * For query (b,t) and head h, over the slots
 *   window rows      max(0, t-W+1) .. t
 *   compressed rows  sq + idx[b,t,s] for every s with 0 <= idx < n_c and
 *                    idx < vis(t) (other entries are padding; a repeated
 *                    entry is a repeated term),
 *   s_i = scale * q[b,t,h,:] . kv_full[b,row_i,:]
 *   lse[b,t,h] = log(exp(sink[h]) + sum_i exp(s_i))
 *   o[b,t,h,:] = sum_i exp(s_i - lse) * kv_full[b,row_i,:]
 * idx == NULL selects every visible block (dense compressed mode); K is then
 * ignored.  fp32 softmax and accumulation; o is cast once to dt.
 * doc_ids ([b, sq] int32, NULL = one document): packed documents ("Refactor
 * Deepseek v4 ...", doc_ids isolation) - a window row k is kept only when
 * doc_ids[b,k] == doc_ids[b,t]; the compressed entries are taken as given
 * (the indexer called with the same doc_ids selects only the query's own
 * document).
 * Errors: INVALID_ARG (null/misaligned pointers, d % 8, window < 1,
 * H < 1, K < 0, n_c != sq / ratio); UNSUPPORTED (d > 512, H > 64).
 */
csa_status_t csa_attn_fwd(const void* q, const void* kv_full, const int32_t* idx,
                          const float* sink, const int32_t* doc_ids, float scale, void* o,
                          float* lse,
                          int b, int sq, int H, int d, int n_c, int ratio, int window, int K,
                          csa_dtype_t dt, csa_stream_t stream);

/*
 * csa_attn_bwd - gradients of the forward above.
 *
 * With D = sum_c dO*o, p_i = exp(s_i - lse), ds_i = p_i (dO . kv_i - D):
 *   dq[b,t,h,:]   = scale * sum_i ds_i kv_i
 *   dkv[b,row,:] += sum over (t,h,slot i with row_i == row) of
 *                   p_i dO[b,t,h,:] + scale ds_i q[b,t,h,:]
 *   dsink[h]      = - sum_{b,t} exp(sink[h] - lse[b,t,h]) * D[b,t,h]
 * The scatter into the compact [b, n_kv, d] buffer accumulates in fp32 and
 * sums repeated indices ("Add unfused SBHD compressed sparse attention",
 * review of the gather backward; "Add the min-memory DSA attention
 * kernels", fp32 scatter).  No [b, sq, n_kv, d] buffer exists.
 * o and lse are the forward's outputs.  dq [b,sq,H,d], dkv [b,n_kv,d] and
 * dsink [H] are fp32 and fully written (dkv and dsink are zeroed by the
 * call).  dsink may be NULL when sink is NULL.  The fp32 atomic sums make
 * dkv and dsink reproducible to rounding only, not bit-for-bit.
 * Errors: as csa_attn_fwd.
 */
csa_status_t csa_attn_bwd(const void* q, const void* kv_full, const int32_t* idx,
                          const float* sink, const int32_t* doc_ids, float scale,
                          const void* o, const float* lse,
                          const void* dO, float* dq, float* dkv, float* dsink,
                          int b, int sq, int H, int d, int n_c, int ratio, int window, int K,
                          csa_dtype_t dt, csa_stream_t stream);

/*
 * Row-range calls: one layer split by query rows across GPUs.
 *
 * The layer partitions by query rows: every query's indexer row, top-k and
 * attention read only shared inputs (kv_full, k_idx, sink), so a GPU that
 * holds those can process any subset of the query rows, and the backward's
 * only cross-row result is the scatter into dkv and dsink, which sums.  The
 * pages keep the sink per head and reject splitting heads across ranks
 * ("Add unfused SBHD compressed sparse attention", attention-sink parameter
 * and the review of its tensor-parallel guard), which leaves the query rows
 * as the axis to split.  These calls take the same arguments as
 * csa_indexer_topk / csa_attn_fwd / csa_attn_bwd, with the full-size arrays
 * (positions stay absolute), plus the query rows [t_begin, t_end) of every
 * batch element to process (0 <= t_begin < t_end <= sq); other rows of the
 * outputs are not touched.
 *
 * csa_attn_bwd_rows: dq rows in the range are written; the range's
 * contributions to dkv and dsink are added to what they hold when
 * accumulate != 0, else dkv and dsink are zeroed first.  The layer's dkv and
 * dsink are the sum of the contributions of disjoint ranges that cover all
 * rows (on one GPU: calls with accumulate = 1 after the first; across GPUs:
 * one sum-reduction of [dkv, dsink]).
 * Errors: as the full calls, plus INVALID_ARG for a range outside [0, sq).
 */
csa_status_t csa_indexer_topk_rows(const void* q_idx, const void* k_idx, const float* w,
                                   const int32_t* doc_ids, int32_t* topk_idx, float* topk_score,
                                   int b, int sq, int n_c, int H_I, int d_I, int ratio, int topk,
                                   csa_dtype_t dt, void* workspace, size_t workspace_bytes,
                                   int t_begin, int t_end, csa_stream_t stream);
csa_status_t csa_attn_fwd_rows(const void* q, const void* kv_full, const int32_t* idx,
                               const float* sink, const int32_t* doc_ids, float scale, void* o,
                               float* lse, int b, int sq, int H, int d, int n_c, int ratio,
                               int window, int K, csa_dtype_t dt, int t_begin, int t_end,
                               csa_stream_t stream);
csa_status_t csa_attn_bwd_rows(const void* q, const void* kv_full, const int32_t* idx,
                               const float* sink, const int32_t* doc_ids, float scale,
                               const void* o, const float* lse, const void* dO, float* dq,
                               float* dkv, float* dsink, int b, int sq, int H, int d, int n_c,
                               int ratio, int window, int K, csa_dtype_t dt, int t_begin,
                               int t_end, int accumulate, csa_stream_t stream);

/*
 * csa_indexer_teacher - distillation target of the indexer.
 *
 * "Refactor Deepseek v4 to use Attention Gym's Compressed Sparse Attention"
 * (indexer distillation): for query (b,t) and each slot s of its index row
 * whose entry j is valid (0 <= j < n_c, j < vis(t)),
 *   T[s] = sum_h exp(scale * q[b,t,h,:] . kv_full[b, sq+j, :] - lse[b,t,h])
 * and target[b,t,:] = T / sum_s T (the teacher is detached: no gradient).
 * lse is the attention forward's LSE (window, selected entries and sink in
 * the denominator).  One common shift per row ("Add unfused SBHD compressed
 * sparse attention", review of the teacher normalization) keeps the mass
 * from underflowing; it cancels in the normalization.  Invalid slots and
 * rows without valid slots hold 0.  A repeated entry gets the same value at
 * each of its slots.
 *
 *   q        in  [b, sq, H, d] dt      kv_full in [b, sq+n_c, d] dt
 *   idx      in  [b, sq, K] int32      lse     in [b, sq, H] fp32
 *   target   out [b, sq, K] fp32
 * Errors: INVALID_ARG (null/misaligned pointers, d % 8, K < 1,
 * n_c != sq / ratio); UNSUPPORTED (d > 512, H > 64, K too large for the
 * kernel's shared memory).
 */
csa_status_t csa_indexer_teacher(const void* q, const void* kv_full, const int32_t* idx,
                                 const float* lse, float scale, float* target, int b, int sq,
                                 int H, int d, int n_c, int ratio, int K, csa_dtype_t dt,
                                 csa_stream_t stream);

/*
 * csa_indexer_loss - the indexer's KL distillation loss over its selected
 * entries, and the gradients through a rescoring of those entries.
 *
 * Student ("Refactor Deepseek v4 ...", lightning indexer: a second pass over
 * the selected entries only): for each valid slot s of query (b,t),
 *   I[s] = sum_h w[b,t,h] * max(0, q_idx[b,t,h,:] . k_idx[b, idx[b,t,s], :]).
 * loss[b,t] = sum_s target[s] * (log target[s] - log softmax(I)[s]) over the
 * valid slots with target > 0; dI = softmax(I) * sum(target) - target ("Add
 * unfused SBHD compressed sparse attention", review of the teacher
 * normalization: a row without mass gets no gradient).  With
 * G[h,s] = dI[s] w[h] [q_idx[h] . k_idx[j_s] > 0]:
 *   dq_idx[b,t,h,:] = sum_s G[h,s] k_idx[j_s]
 *   dw[b,t,h]       = sum_s dI[s] max(0, q_idx[h] . k_idx[j_s])
 *   dk_idx[b,j,:]  += sum over (t, s with j_s = j) sum_h G[h,s] q_idx[b,t,h]
 * All outputs fp32; dk_idx is zeroed by the call and accumulated with fp32
 * atomics (reproducible to rounding only).  target is usually the output of
 * csa_indexer_teacher for the same idx.
 *
 *   q_idx [b,sq,H_I,d_I] dt  k_idx [b,n_c,d_I] dt  w [b,sq,H_I] fp32
 *   idx [b,sq,K] int32  target [b,sq,K] fp32
 *   loss out [b,sq]  dq_idx out [b,sq,H_I,d_I]  dk_idx out [b,n_c,d_I]
 *   dw out [b,sq,H_I]
 * Errors: INVALID_ARG (null/misaligned pointers, d_I % 8, K < 1,
 * n_c != sq / ratio); UNSUPPORTED (d_I > 256, H_I > 64, K too large).
 */
csa_status_t csa_indexer_loss(const void* q_idx, const void* k_idx, const float* w,
                              const int32_t* idx, const float* target, float* loss,
                              float* dq_idx, float* dk_idx, float* dw, int b, int sq, int n_c,
                              int H_I, int d_I, int ratio, int K, csa_dtype_t dt,
                              csa_stream_t stream);

/*
 * Read and clear the device status word of the current device after the
 * work on `stream` has finished (this call synchronizes `stream`).
 * *status_out receives CSA_OK, CSA_ERR_TIMEOUT or CSA_ERR_DEVICE_CHECK (the
 * first error recorded since the last read).  site_out (nullable) receives
 * where it was recorded:
 *   CSA_ERR_TIMEOUT: 0x11-0x13 the indexer's TMA producer, MMA issuer or
 *   epilogue waits; 0x21-0x24 the tensor-core attention forward's waits for
 *   the Q tile, the score MMA, the PV MMA inside the loop and the last PV
 *   MMA (the d = 512 forward records the same sites); 0x31-0x34 the
 *   tensor-core backward's waits for the Q/dO tiles, the S/dP MMAs, the P^T dO
 *   MMAs and the dS MMAs (the d = 512 backward: 0x31 its Q/dO/KV stages, 0x32
 *   and 0x34 its products); 0x51-0x53 the tensor-core indexer loss's waits
 *   for the q_idx tile, the dots X^T and the dq_idx / dk_idx products;
 *   0x61-0x62 the tensor-core indexer teacher's waits for the Q tile and the
 *   transposed scores S^T.
 *   CSA_ERR_DEVICE_CHECK: 0x25 the tensor-core forward found the union of a
 *   query block's selected blocks larger than its n_c-entry list; 0x41 a
 *   packed document (doc_ids of csa_indexer_topk / csa_indexer_topk_fp8)
 *   starts inside a compressed block (documents must start on multiples of
 *   ratio; the results follow the rule that a block belongs to the document
 *   of its first token).
 * Every device wait of the library is bounded (about one second of wall
 * time); a wait that gives up records CSA_ERR_TIMEOUT here and its CTA skips
 * the rest of its work, as does a CTA whose check at 0x25 fails, so the
 * results of that call are not valid.
 */
csa_status_t csa_get_device_status(csa_stream_t stream, int* status_out, int* site_out);

/*
 * csa_debug_arm_fault - test hook of the failure-detection paths (not part
 * of the method; the pages have no counterpart).
 *
 * With site = 0x21 every later tensor-core attention forward on the current
 * device never requests its Q tile, so its bounded wait runs out (about one
 * second) with no copy or MMA in flight and records CSA_ERR_TIMEOUT at 0x21;
 * with site = 0x25 its union-size check trips and records
 * CSA_ERR_DEVICE_CHECK at 0x25.  site = 0 disarms.  The call synchronizes
 * the device.  Use it only in tests.
 * Errors: INVALID_ARG for site < 0; CSA_ERR_CUDA if the device is unusable.
 */
csa_status_t csa_debug_arm_fault(int site);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
