// Low-bit cache formats ("DeepSeek V4.1 Flash", production cache ABI): packed
// E2M1 with E4M3 group-of-16 scales (compressed KV), packed E2M1 with E8M0
// group-of-32 scales (index keys) and MXFP8 (E4M3 with E8M0 group-of-32
// scales, window KV).  Two E2M1 codes share a byte, channel 2i in the low
// nibble.  Publication rounds as include/csa.h states; reads decode exactly.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "csa_internal.cuh"

namespace csa {
namespace lowbit {

// E2M1 code (sign | 3-bit magnitude code) of the representable value
// nearest to x: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 for codes 0..7; a value
// halfway between two goes to the even code; above 6 saturates.
__device__ __forceinline__ uint32_t e2m1_code(float x) {
  const float a = fabsf(x);
  uint32_t m;
  if (a <= 0.25f) m = 0;        // 0.25: tie 0 / 0.5 -> 0
  else if (a < 0.75f) m = 1;
  else if (a <= 1.25f) m = 2;   // 0.75: 0.5 / 1 -> 1; 1.25: 1 / 1.5 -> 1
  else if (a < 1.75f) m = 3;
  else if (a <= 2.5f) m = 4;    // 1.75: 1.5 / 2 -> 2; 2.5: 2 / 3 -> 2
  else if (a < 3.5f) m = 5;
  else if (a <= 5.0f) m = 6;    // 3.5: 3 / 4 -> 4; 5: 4 / 6 -> 4
  else m = 7;
  return m | (x < 0.f ? 8u : 0u);
}

// The E8M0 exponent of a group: the smallest e with 6 * 2^e >= amax, in
// [-127, 127] (amax = 0: -127).  With amax = m * 2^k, m in [0.5, 1):
// amax = (2m) * 2^(k-1) and e = k - 3 + (2m > 1.5).
__device__ __forceinline__ int e8m0_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  int k;
  const float m = frexpf(amax, &k);
  const int e = k - 3 + (2.f * m > 1.5f ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// The E4M3 scale byte of a group (nearest E4M3 to amax / 6, saturating) and
// its value.
__device__ __forceinline__ uint32_t e4m3_scale_byte(float amax) {
  return (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(amax, 6.f), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_value(uint32_t byte) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3);
  return __half2float(__half(h));
}

// Two E2M1 codes (one byte, channel 2i in the low nibble) as an FP16 pair
// (channel 2i in the low half): the sm_100-family conversion instruction.
__device__ __forceinline__ uint32_t cvt_e2m1x2(uint32_t byte) {
  uint32_t d;
  const uint16_t v = (uint16_t)(byte & 0xFFu);
  asm("{\n .reg .b8 b;\n cvt.u8.u16 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(d) : "h"(v));
  return d;
}
// Two E4M3 codes (the low byte first) as an FP16 pair (low half first).
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two) {
  uint32_t d;
  const uint16_t v = (uint16_t)(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<const __half2 *>(&u); }

// 2^e as a float for e in [-127, 127] (2^-127 is an FP32 subnormal).
__device__ __forceinline__ float pow2f(int e) { return ldexpf(1.f, e); }

// 2^s as an FP16 pair for s <= 0: exact down to 2^-24 (subnormal), 0 below.
__device__ __forceinline__ __half2 pow2_h2(int s) {
  uint16_t bits = 0;
  if (s >= -14)
    bits = (uint16_t)((s + 15) << 10);
  else if (s >= -24)
    bits = (uint16_t)(1u << (s + 24));
  const __half h = __ushort_as_half(bits);
  return __halves2half2(h, h);
}

// Eight E2M1 codes (one word; byte i holds channels 2i (low nibble) and
// 2i+1) as eight FP16 values times `scale2` (a power of two: the products
// are exact unless they fall below 2^-24).
__device__ __forceinline__ uint4 e2m1x8_to_f16x8(uint32_t w, __half2 scale2) {
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __hmul2(as_h2(cvt_e2m1x2(w >> (8 * i))), scale2);
    out[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Eight E4M3 codes (two words, the low byte first) as eight FP16 values
// times `scale2` (a power of two; exact unless a product falls below 2^-24).
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 w, __half2 scale2) {
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t word = i < 2 ? w.x : w.y;
    const __half2 h = __hmul2(as_h2(cvt_e4m3x2(word >> (16 * (i & 1)))), scale2);
    out[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// The E8M0 exponent of an MXFP8 group: the smallest e with 448 * 2^e >=
// amax, in [-127, 127] (amax = 0: -127).  With amax = m * 2^k, m in
// [0.5, 1): e = k - 9 + (2m > 1.75).
__device__ __forceinline__ int e8m0_exponent_448(float amax) {
  if (!(amax > 0.f)) return -127;
  int k;
  const float m = frexpf(amax, &k);
  const int e = k - 9 + (2.f * m > 1.75f ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Row shift of an FP4 index key: R = the largest of its four E8M0 exponents
// (scale bytes in one word).  The key's values are dequantised to FP16 as
// code * 2^(E_g - R), and 2^R multiplies the key's score.
__device__ __forceinline__ int e8m0_row_shift(uint32_t sb4) {
  const int e0 = (int)(sb4 & 0xFFu), e1 = (int)((sb4 >> 8) & 0xFFu);
  const int e2 = (int)((sb4 >> 16) & 0xFFu), e3 = (int)(sb4 >> 24);
  return max(max(e0, e1), max(e2, e3)) - 127;
}
__device__ __forceinline__ __half2 e8m0_group_h2(uint32_t sb4, int g, int R) {
  return pow2_h2((int)((sb4 >> (8 * g)) & 0xFFu) - 127 - R);
}

// Eight FP4 channels (one word of E2M1 codes) times an E4M3 scale, as eight
// BF16 values.  The product of an E2M1 and an E4M3 value has at most six
// significant bits and lies in [2^-10, 2688]: exact in FP16 and in BF16.
__device__ __forceinline__ uint4 e2m1x8_e4m3_to_bf16x8(uint32_t w, uint32_t sbyte) {
  const __half2 s2 = __half2half2(__low2half(as_h2(cvt_e4m3x2(sbyte))));
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(__hmul2(as_h2(cvt_e2m1x2(w >> (8 * i))), s2));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    out[i] = *reinterpret_cast<const uint32_t *>(&b);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Eight MXFP8 channels (two words of E4M3 codes) times their E8M0 scale, as
// eight BF16 values (exact: an E4M3 value has four significant bits).
__device__ __forceinline__ uint4 e4m3x8_e8m0_to_bf16x8(uint2 w, float scale) {
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t word = i < 2 ? w.x : w.y;
    const float2 f = __half22float2(as_h2(cvt_e4m3x2(word >> (16 * (i & 1)))));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    out[i] = *reinterpret_cast<const uint32_t *>(&b);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace lowbit
}  // namespace csa
