// Element loads for the attention kernels (fp32 / bf16 / fp8 e4m3 storage).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bd {

// Four consecutive elements starting at element index i (i % 4 == 0) as fp32.
// E4M3 values are returned unscaled: the per-head scales are applied to the
// scores (K) and to the merged output (V).
template <int DT>
__device__ __forceinline__ float4 load4(const void* base, size_t i);

template <>
__device__ __forceinline__ float4 load4<0>(const void* base, size_t i) {
  return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
}
template <>
__device__ __forceinline__ float4 load4<1>(const void* base, size_t i) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + i));
  float4 f;
  f.x = __uint_as_float(u.x << 16);
  f.y = __uint_as_float(u.x & 0xffff0000u);
  f.z = __uint_as_float(u.y << 16);
  f.w = __uint_as_float(u.y & 0xffff0000u);
  return f;
}
template <>
__device__ __forceinline__ float4 load4<2>(const void* base, size_t i) {
  const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(static_cast<const uint8_t*>(base) + i));
  __nv_fp8x2_storage_t lo = (__nv_fp8x2_storage_t)(u & 0xffffu);
  __nv_fp8x2_storage_t hi = (__nv_fp8x2_storage_t)(u >> 16);
  const float2 a = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
  const float2 b = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void store_out4(void* out, size_t i, float4 v, int out_dtype) {
  if (out_dtype == 0) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = v;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + i) = u;
  }
}

}  // namespace bd
