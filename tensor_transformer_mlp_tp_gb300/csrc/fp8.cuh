// E4M3 helpers: the saturating round-to-nearest cast of CUDA's cuda_fp8.h, the
// float32 product x * s formed first (round to nearest), and the amax combine.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace tpmlp {

// E4M3(a s), E4M3(b s), E4M3(c s), E4M3(d s) in one word, the first value in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float s) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(a, s), __fmul_rn(b, s)), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(c, s), __fmul_rn(d, s)), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

__device__ __forceinline__ uint2 e4m3x8(const float (&f)[8], float s) {
  return make_uint2(e4m3x4(f[0], f[1], f[2], f[3], s), e4m3x4(f[4], f[5], f[6], f[7], s));
}

// The same for E5M2 (the gradients' format: 2 mantissa bits, saturating at +-57344).
__device__ __forceinline__ uint32_t e5m2x4(float a, float b, float c, float d, float s) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(a, s), __fmul_rn(b, s)), __NV_SATFINITE, __NV_E5M2);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(c, s), __fmul_rn(d, s)), __NV_SATFINITE, __NV_E5M2);
  return lo | (hi << 16);
}

// FMT 0 = E4M3, 1 = E5M2.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d, float s) {
  if constexpr (FMT == 0) {
    return e4m3x4(a, b, c, d, s);
  } else {
    return e5m2x4(a, b, c, d, s);
  }
}

template <int FMT>
__device__ __forceinline__ uint2 fp8x8(const float (&f)[8], float s) {
  return make_uint2(fp8x4<FMT>(f[0], f[1], f[2], f[3], s), fp8x4<FMT>(f[4], f[5], f[6], f[7], s));
}

// Max-combine a warp's values into *amax (all lanes call it).  Non-negative floats order like their bit
// patterns, so an integer max combines them; a lane whose value does not exceed what *amax already
// holds skips the atomic.
__device__ __forceinline__ void amax_combine_warp(float* amax, float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0 && m > *reinterpret_cast<volatile float*>(amax))
    atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
}

}  // namespace tpmlp
