// Per-row e4m3 codes of bf16 values, shared by the quantisation kernel
// (quant.cu) and the gather that writes codes directly (gather.cu), so that
// both give the same bytes: s = amax / 448 (448 = the largest finite e4m3
// value), q = e4m3(x * (448 / amax)) rounded to nearest even and saturated,
// both quotients IEEE binary32 divisions; an all-zero row gets s = 1 and zero
// codes.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace engram {
namespace e4m3 {

constexpr float kMax = 448.f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// two values -> two codes in one conversion: a in the low byte, b in the high byte
__device__ __forceinline__ uint32_t bytes2_of(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// the largest |x| of eight bf16 values (a 16-byte chunk), folded into amax
__device__ __forceinline__ float amax8(uint4 v, float amax) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  return amax;
}

__device__ __forceinline__ float inv_of(float amax) { return amax > 0.f ? kMax / amax : 0.f; }
__device__ __forceinline__ float scale_of(float amax) { return amax > 0.f ? amax / kMax : 1.f; }

// eight bf16 values times inv -> eight codes, element j in byte j
__device__ __forceinline__ uint2 quant8(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 4; ++j) out[j >> 1] |= bytes2_of(bf16_lo(w[j]) * inv, bf16_hi(w[j]) * inv) << ((j & 1) * 16);
  return make_uint2(out[0], out[1]);
}

}  // namespace e4m3
}  // namespace engram
