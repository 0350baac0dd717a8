// OCP MX quantisation of activations to MXFP4 (OCP Microscaling Formats (MX)
// Specification v1.0): 32-element blocks along K, shared scale
// X = 2^(floor(log2 amax) - 2) stored as an E8M0 byte clamped to [0, 254]
// (2^-127 for an all-zero block), each element the E2M1 value nearest to
// v / X with ties to the even code, saturated at 6, +0 for a zero magnitude.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace moe {

// E8M0 byte of the shared scale from the block's largest magnitude.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  const uint32_t e = (__float_as_uint(amax) >> 23) & 0xffu;  // biased exponent; 0 for zero and subnormals
  return e > 2u ? e - 2u : 0u;                                // floor(log2 amax) - 2 + 127, clamped at 0
}

// 1 / X as a float (exact power of two; byte <= 252 for finite inputs).
__device__ __forceinline__ float mx_inv_scale(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }

// X as a float (2^-127 is a subnormal).
__device__ __forceinline__ float mx_scale(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// E2M1 code (0..15) of v / X: nearest grid value, ties to the even code.
__device__ __forceinline__ uint32_t mx_code(float v, float inv_x) {
  const float m = fabsf(v) * inv_x;  // exact: inv_x is a power of two
  const uint32_t c = (uint32_t)(m > 0.25f) + (uint32_t)(m >= 0.75f) + (uint32_t)(m > 1.25f) +
                     (uint32_t)(m >= 1.75f) + (uint32_t)(m > 2.5f) + (uint32_t)(m >= 3.5f) + (uint32_t)(m > 5.f);
  return (c != 0u && v < 0.f) ? (c | 8u) : c;
}

// The value an E2M1 code stands for, times X (exact in fp32 and in bf16).
__device__ __forceinline__ float mx_value(uint32_t code, float x_scale) {
  const uint32_t m = code & 7u, e = m >> 1, mant = m & 1u;
  const float mag = e ? __uint_as_float(((e + 126u) << 23) | (mant << 22)) : 0.5f * (float)mant;
  return ((code & 8u) ? -mag : mag) * x_scale;
}

// Activations of the block-scaled decode GEMM: a 32-element block along K
// shares a power-of-two scale X = 2^(floor(log2 amax) - 7), which puts the
// block's largest magnitude in [128, 256), below E4M3's largest finite value
// (448); each scaled value v / X is carried as two E4M3 terms, hi = E4M3(v / X)
// and lo = E4M3(v / X - hi), both rounded to nearest even.  hi + lo holds
// eight significant bits of v / X (a bf16 input exactly, unless lo falls
// below E4M3's normal range).  The scale byte is clamped to [0, 247], so 1 / X
// stays a normal float.
__device__ __forceinline__ uint32_t mx8_scale_byte(float amax) {
  const uint32_t e = (__float_as_uint(amax) >> 23) & 0xffu;
  return e > 7u ? (e - 7u < 247u ? e - 7u : 247u) : 0u;
}

// Two values -> an E4M3 pair (v0 in the low byte), nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2_rn(float v0, float v1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v1), "f"(v0));
  return r;
}

// An E4M3 pair (low byte first) -> two floats (exact).
__device__ __forceinline__ void e4m3x2_f32(uint32_t two, float& v0, float& v1) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
  v0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
  v1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// hi and lo E4M3 pairs of two scaled values (v0 in the low bytes).  v - hi is
// exact in fp32 (hi is v rounded to four significant bits).
__device__ __forceinline__ void mx8_split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  hi = e4m3x2_rn(v0, v1);
  float h0, h1;
  e4m3x2_f32(hi, h0, h1);
  lo = e4m3x2_rn(v0 - h0, v1 - h1);
}

}  // namespace moe
