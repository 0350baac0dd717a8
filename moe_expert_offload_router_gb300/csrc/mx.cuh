// OCP MX quantisation of activations to MXFP4 (OCP Microscaling Formats (MX)
// Specification v1.0): 32-element blocks along K, shared scale
// X = 2^(floor(log2 amax) - 2) stored as an E8M0 byte clamped to [0, 254]
// (2^-127 for an all-zero block), each element the E2M1 value nearest to
// v / X with ties to the even code, saturated at 6, +0 for a zero magnitude.
#pragma once

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

}  // namespace moe
