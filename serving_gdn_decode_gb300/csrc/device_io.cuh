// Device-side staging and element access shared by the token-loop and scan
// kernels: cp.async into shared memory, and reads/writes of the activation
// buffers (q, k, v, output) as f32 or as bf16 widened to f32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gdn {

__device__ __forceinline__ void cp_async_16(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_4(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Activation element type: f32, or bf16 (exact widening on read; one
// round-to-nearest-even on write).
template <typename IO>
struct Act;

template <>
struct Act<float> {
  static constexpr int kPer4B = 1;  // elements per 4-byte cp.async
  static __device__ __forceinline__ float get(const float *p) { return *p; }
  static __device__ __forceinline__ void put(float *p, float x) { *p = x; }
  // n contiguous elements from shared memory (n = 1, 2 or 4; p aligned to n elements)
  template <int N>
  static __device__ __forceinline__ void get_n(const float *p, float *c) {
    if constexpr (N == 4) {
      const float4 x = *reinterpret_cast<const float4 *>(p);
      c[0] = x.x; c[1] = x.y; c[2] = x.z; c[3] = x.w;
    } else if constexpr (N == 2) {
      const float2 x = *reinterpret_cast<const float2 *>(p);
      c[0] = x.x; c[1] = x.y;
    } else {
      c[0] = *p;
    }
  }
};

template <>
struct Act<__nv_bfloat16> {
  static constexpr int kPer4B = 2;
  static __device__ __forceinline__ float get(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void put(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
  template <int N>
  static __device__ __forceinline__ void get_n(const __nv_bfloat16 *p, float *c) {
    if constexpr (N == 4) {
      const uint2 w = *reinterpret_cast<const uint2 *>(p);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
      c[0] = lo.x; c[1] = lo.y; c[2] = hi.x; c[3] = hi.y;
    } else if constexpr (N == 2) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
      c[0] = x.x; c[1] = x.y;
    } else {
      c[0] = __bfloat162float(*p);
    }
  }
};

}  // namespace gdn
