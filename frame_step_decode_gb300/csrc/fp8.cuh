// fp8.cuh -- E4M3 encode/decode of the K/V cache (OCP 8-bit floating point,
// E4M3 variant: bias 7, no infinities, S.1111.111 = NaN, max finite 448).
//
// Encode: hardware conversion, round to nearest even, saturating to +-448
// (cuda_fp8.h intrinsic).  Decode: hardware paired conversion to f16, which
// is exact because every E4M3 value is an f16 value.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace wave {

__device__ __forceinline__ uint8_t e4m3_encode(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Two codes in the low/high byte of a 16-bit word -> f16x2 (low half = low byte).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Four codes in a 32-bit word -> two f16x2: lo = bytes 0,1, hi = bytes 2,3
// (byte k of each pair in half k).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Per-row quantiser of the K/V append (one warp, D = 32 * kPer values, lane
// i holding elements [i*kPer, (i+1)*kPer)): scale = amax/448 (fp32, RN),
// codes = E4M3(v / scale) with an IEEE fp32 division; a zero row gives
// all-zero codes and scale 0.  Returns the lane's codes packed little-endian.
template <int kPer>
__device__ __forceinline__ uint32_t quantize_lane(const float* v, float& scale_out) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float s = __fdiv_rn(amax, 448.0f);
  scale_out = s;
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    uint32_t c = (s == 0.f) ? 0u : (uint32_t)e4m3_encode(__fdiv_rn(v[i], s));
    packed |= c << (8 * i);
  }
  return packed;
}

}  // namespace wave
