// Sparse MQA forward/backward on CUDA cores: the exact-fp32 path (fp32
// inputs) and the generic path for shapes the tensor-core kernels do not
// cover.  One CTA per query row, one warp per head, online softmax.
//
// Semantics ("Add unfused SBHD compressed sparse attention": unfused sparse
// core, sink parameter, review of the gather backward; "Refactor Deepseek v4
// to use Attention Gym's Compressed Sparse Attention": window + selected
// entries + sink in one softmax with per-head LSE):
//   slots = window rows max(0,t-W+1)..t, then sq+j for valid idx entries
//   s_i = scale q.kv_i; lse = log(e^sink + sum e^s_i); o = sum e^(s_i-lse) kv_i
//   bwd: D = dO.o, p_i = e^(s_i-lse), ds_i = p_i (dO.kv_i - D),
//        dq = scale sum ds_i kv_i, dkv_i += p_i dO + scale ds_i q,
//        dsink = -e^(sink-lse) D.
#include "csa_common.cuh"
#include "csa_kernels.h"

namespace csa {

constexpr int kSimtWarps = 4;
constexpr int kMaxPerLane = 16;  // d <= 512

template <typename T>
__global__ void __launch_bounds__(128) attn_fwd_simt(const T* __restrict__ q,
                                                     const T* __restrict__ kv,
                                                     const int32_t* __restrict__ idx,
                                                     const float* __restrict__ sink, float scale,
                                                     T* __restrict__ o, float* __restrict__ lse,
                                                     int sq, int H, int d, int n_c, int ratio,
                                                     int window, int K,
                                                     const int32_t* __restrict__ doc, int tb) {
  extern __shared__ int rows[];
  const int t = tb + (int)blockIdx.x, bi = blockIdx.y;
  const int wid = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int n_kv = sq + n_c;
  __shared__ int s_count;
  if (wid == 0) {
    const int c = build_slots_warp(rows, idx ? idx + ((long long)bi * sq + t) * K : nullptr, K, t,
                                   sq, n_c, ratio, window, doc ? doc + (long long)bi * sq : nullptr);
    if (lane == 0) s_count = c;
  }
  __syncthreads();
  const int count = s_count;
  const int per = (d + 31) / 32;
  const float sc2 = scale * kLog2e;
  for (int h = wid; h < H; h += kSimtWarps) {
    const T* qh = q + (((long long)bi * sq + t) * H + h) * d;
    float qv[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int c = lane + 32 * i;
      qv[i] = (i < per && c < d) ? to_f(qh[c]) : 0.f;
      acc[i] = 0.f;
    }
    float m = sink ? sink[h] * kLog2e : -INFINITY;
    float l = sink ? 1.f : 0.f;
    for (int s = 0; s < count; ++s) {
      const T* kr = kv + ((long long)bi * n_kv + rows[s]) * d;
      float kvv[kMaxPerLane];
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        kvv[i] = (i < per && c < d) ? to_f(kr[c]) : 0.f;
        part = fmaf(qv[i], kvv[i], part);
      }
      const float s2 = warp_sum(part) * sc2;
      const float mn = fmaxf(m, s2);
      const float alpha = exp2f(m - mn);
      const float p = exp2f(s2 - mn);
      l = l * alpha + p;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) acc[i] = fmaf(acc[i], alpha, p * kvv[i]);
      m = mn;
    }
    T* oh = o + (((long long)bi * sq + t) * H + h) * d;
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int c = lane + 32 * i;
      if (i < per && c < d) oh[c] = from_f<T>(acc[i] * inv);
    }
    if (lane == 0) lse[((long long)bi * sq + t) * H + h] = (m + log2f(l)) * kLn2;
  }
}

template <typename T>
__global__ void __launch_bounds__(128) attn_bwd_simt(
    const T* __restrict__ q, const T* __restrict__ kv, const int32_t* __restrict__ idx,
    const float* __restrict__ sink, float scale, const T* __restrict__ o,
    const float* __restrict__ lse, const T* __restrict__ dO, float* __restrict__ dq,
    float* __restrict__ dkv, float* __restrict__ dsink, int sq, int H, int d, int n_c, int ratio,
    int window, int K, const int32_t* __restrict__ doc, int tb) {
  extern __shared__ int rows[];
  const int t = tb + (int)blockIdx.x, bi = blockIdx.y;
  const int wid = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int n_kv = sq + n_c;
  __shared__ int s_count;
  if (wid == 0) {
    const int c = build_slots_warp(rows, idx ? idx + ((long long)bi * sq + t) * K : nullptr, K, t,
                                   sq, n_c, ratio, window, doc ? doc + (long long)bi * sq : nullptr);
    if (lane == 0) s_count = c;
  }
  __syncthreads();
  const int count = s_count;
  const int per = (d + 31) / 32;
  const float sc2 = scale * kLog2e;
  for (int h = wid; h < H; h += kSimtWarps) {
    const long long base = (((long long)bi * sq + t) * H + h) * d;
    float qv[kMaxPerLane], gv[kMaxPerLane], dqa[kMaxPerLane];
    float dpart = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int c = lane + 32 * i;
      const bool ok = i < per && c < d;
      qv[i] = ok ? to_f(q[base + c]) : 0.f;
      gv[i] = ok ? to_f(dO[base + c]) : 0.f;
      dpart = fmaf(gv[i], ok ? to_f(o[base + c]) : 0.f, dpart);
      dqa[i] = 0.f;
    }
    const float Dh = warp_sum(dpart);
    const float L = lse[((long long)bi * sq + t) * H + h];
    const float lse2 = L * kLog2e;
    if (sink && lane == 0) atomicAdd(&dsink[h], -exp2f(sink[h] * kLog2e - lse2) * Dh);
    for (int s = 0; s < count; ++s) {
      float* dkr = dkv + ((long long)bi * n_kv + rows[s]) * d;
      const T* kr = kv + ((long long)bi * n_kv + rows[s]) * d;
      float kvv[kMaxPerLane];
      float ps = 0.f, pp = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        kvv[i] = (i < per && c < d) ? to_f(kr[c]) : 0.f;
        ps = fmaf(qv[i], kvv[i], ps);
        pp = fmaf(gv[i], kvv[i], pp);
      }
      const float s2 = warp_sum(ps) * sc2;
      const float dp = warp_sum(pp);
      const float p = exp2f(s2 - lse2);
      const float ds = p * (dp - Dh);
      const float sds = scale * ds;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        if (i < per && c < d) {
          dqa[i] = fmaf(sds, kvv[i], dqa[i]);
          atomicAdd(&dkr[c], fmaf(p, gv[i], sds * qv[i]));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int c = lane + 32 * i;
      if (i < per && c < d) dq[base + c] = dqa[i];
    }
  }
}

cudaError_t launch_attn_fwd_simt(const void* q, const void* kv, const int32_t* idx,
                                 const float* sink, float scale, void* o, float* lse, int b,
                                 int sq, int H, int d, int n_c, int ratio, int window, int K,
                                 bool bf16, cudaStream_t s, const int32_t* doc, int tb, int te) {
  dim3 grid((unsigned)(te - tb), (unsigned)b);
  const size_t smem = (size_t)(window + (idx ? K : n_c) + 32) * sizeof(int);
  if (bf16) {
    attn_fwd_simt<__nv_bfloat16><<<grid, 32 * kSimtWarps, smem, s>>>(
        (const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx, sink, scale, (__nv_bfloat16*)o,
        lse, sq, H, d, n_c, ratio, window, K, doc, tb);
    count_launches(1);
  } else {
    attn_fwd_simt<float><<<grid, 32 * kSimtWarps, smem, s>>>((const float*)q, (const float*)kv,
                                                             idx, sink, scale, (float*)o, lse, sq,
                                                             H, d, n_c, ratio, window, K, doc,
                                                             tb);
    count_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_simt(const void* q, const void* kv, const int32_t* idx,
                                 const float* sink, float scale, const void* o, const float* lse,
                                 const void* dO, float* dq, float* dkv, float* dsink, int b,
                                 int sq, int H, int d, int n_c, int ratio, int window, int K,
                                 bool bf16, cudaStream_t s, const int32_t* doc, int tb, int te) {
  dim3 grid((unsigned)(te - tb), (unsigned)b);
  const size_t smem = (size_t)(window + (idx ? K : n_c) + 32) * sizeof(int);
  if (bf16) {
    attn_bwd_simt<__nv_bfloat16><<<grid, 32 * kSimtWarps, smem, s>>>(
        (const __nv_bfloat16*)q, (const __nv_bfloat16*)kv, idx, sink, scale,
        (const __nv_bfloat16*)o, lse, (const __nv_bfloat16*)dO, dq, dkv, dsink, sq, H, d, n_c,
        ratio, window, K, doc, tb);
    count_launches(1);
  } else {
    attn_bwd_simt<float><<<grid, 32 * kSimtWarps, smem, s>>>(
        (const float*)q, (const float*)kv, idx, sink, scale, (const float*)o, lse,
        (const float*)dO, dq, dkv, dsink, sq, H, d, n_c, ratio, window, K, doc, tb);
    count_launches(1);
  }
  return cudaGetLastError();
}

__global__ void zero_f32_kernel(float4* __restrict__ p, size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}
__global__ void zero_f32_tail(float* __restrict__ p, size_t n) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0.f;
}

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const size_t n4 = n / 4;
  if (n4) {
    size_t blocks = (n4 + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    zero_f32_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<float4*>(p), n4);
    count_launches(1);
  }
  const size_t rem = n - n4 * 4;
  if (rem) {
    zero_f32_tail<<<1, 32, 0, s>>>(p + n4 * 4, rem);
    count_launches(1);
  }
  return cudaGetLastError();
}

// Zero a (na floats, 16-byte aligned, na % 4 == 0) and b (nb floats) in one
// launch: the backward's dkv and dsink.
__global__ void zero_f32_pair_kernel(float4* __restrict__ a, size_t na4, float* __restrict__ b,
                                     size_t nb) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nb) b[i] = 0.f;
  for (; i < na4; i += stride) a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_zero_f32_pair(float* a, size_t na, float* b, size_t nb, cudaStream_t s) {
  if (na % 4 != 0 || nb > 256 * 152) {
    cudaError_t e = launch_zero_f32(a, na, s);
    return e == cudaSuccess ? launch_zero_f32(b, nb, s) : e;
  }
  size_t blocks = (na / 4 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks * 256 < nb) blocks = (nb + 255) / 256;
  if (blocks == 0) return cudaSuccess;
  zero_f32_pair_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<float4*>(a), na / 4, b,
                                                       nb);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
