// Shared device helpers of the CSA CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// Process-wide count of kernels this library has enqueued (every launcher
// adds its launches); read through csa_kernel_launches().
void count_launches(int n);

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status codes (same values as csa_status_t).
constexpr int kDevTimeout = 5;
constexpr int kDevCheck = 6;

// The device status word is two ints: [0] the first error code, [1] the
// site that recorded it (which kernel and which wait), for diagnosis.
__device__ __forceinline__ void set_status(int* status, int code, int site = 0) {
  if (status != nullptr && atomicCAS(status, 0, code) == 0) atomicExch(status + 1, site);
}

// Sites recorded with CSA_ERR_TIMEOUT.
constexpr int kSiteIdxProducer = 0x11, kSiteIdxMma = 0x12, kSiteIdxEpilogue = 0x13;
constexpr int kSiteFwdQ = 0x21, kSiteFwdS = 0x22, kSiteFwdO = 0x23, kSiteFwdLast = 0x24;
constexpr int kSiteBwdQ = 0x31, kSiteBwdS = 0x32, kSiteBwdP = 0x33, kSiteBwdDS = 0x34;
constexpr int kSiteLossQ = 0x51, kSiteLossX = 0x52, kSiteLossG = 0x53;
constexpr int kSiteTeacherQ = 0x61, kSiteTeacherS = 0x62;
// Sites recorded with CSA_ERR_DEVICE_CHECK: the tensor-core forward's union
// of selected blocks larger than its n_c-entry list; a packed document that
// starts inside a compressed block.
constexpr int kSiteFwdUnion = 0x25, kSiteDocBoundary = 0x41;

// The status word's third int holds a test hook (csa_debug_arm_fault): the
// site at which a kernel fakes a failure (0 = none).  Kernels read it once.
__device__ __forceinline__ int armed_fault(const int* status) {
  return status != nullptr ? *(volatile const int*)(status + 2) : 0;
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Load 8 consecutive elements (16 B for bf16, 32 B for fp32) as floats.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* f) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* f) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* f) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float* f) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// Two independent fp32 fused multiply-adds in one instruction (fma.rn.f32x2,
// sm_100 and later): a += w.x * y0, b += w.y * y1, each rounded once to
// nearest exactly as fmaf rounds, so results are bit-identical to two fmaf.
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void fma_f32x2(float& a, float& b, unsigned long long w,
                                          float y0, float y1) {
  unsigned long long acc = pack_f32x2(a, b);
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(w), "l"(pack_f32x2(y0, y1)));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(acc));
}

// fp32 atomic adds into global memory (no return value).
__device__ __forceinline__ void red_add_f32(float* addr, float a) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}
__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
  asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b)
               : "memory");
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Gather the attention slot rows of query t into `rows` (flat kv_full row ids
// within the batch element): window rows max(0,t-W+1)..t (with per-token
// document ids doc_b, only those of t's document), then sq+j for the valid
// entries j of the index row (0 <= j < n_c and j < vis(t)), in index order.
// idx == nullptr means every visible block.  Executed by one warp; returns
// the slot count to every lane.
__device__ __forceinline__ int build_slots_warp(int* rows, const int32_t* idx_row, int K, int t,
                                                int sq, int n_c, int ratio, int window,
                                                const int32_t* doc_b = nullptr) {
  const int lane = threadIdx.x & 31;
  const int w0 = max(0, t - window + 1);
  int nw = t - w0 + 1;
  if (doc_b == nullptr) {
    for (int i = lane; i < nw; i += 32) rows[i] = w0 + i;
  } else {
    const int dt = doc_b[t];
    int kept = 0;
    for (int base = 0; base < nw; base += 32) {
      const int k = w0 + base + lane;
      const bool ok = base + lane < nw && doc_b[k] == dt;
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) rows[kept + __popc(m & ((1u << lane) - 1u))] = k;
      kept += __popc(m);
    }
    nw = kept;
  }
  const int vis = min((t + 1) / ratio, n_c);
  int count = nw;
  if (idx_row == nullptr) {
    for (int j = lane; j < vis; j += 32) rows[nw + j] = sq + j;
    return nw + vis;
  }
  for (int base = 0; base < K; base += 32) {
    const int s = base + lane;
    int j = -1;
    if (s < K) j = idx_row[s];
    const bool ok = (j >= 0) && (j < vis);
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) rows[count + __popc(m & ((1u << lane) - 1u))] = sq + j;
    count += __popc(m);
  }
  return count;
}

}  // namespace csa
