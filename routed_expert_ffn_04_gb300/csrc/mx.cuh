// MXFP8 element helpers (E4M3 elements, E8M0 block scales; OCP MX v1.0):
// the block shared exponent and element encoding of the OCP MX conversion
// rule, and the exact expansion of scaled E4M3 codes into bf16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

__device__ __forceinline__ float pow2f(int e) {  // exact 2^e, -127 <= e <= 127
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Value of one E4M3 code times 2^(sc - 127), as bf16 bits (exact unless the
// product falls below the bf16 range).
__device__ __forceinline__ uint32_t e4m3_scaled_bf16_slow(uint32_t b, int sc) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v;
  if (e == 15u && m == 7u) {
    v = __uint_as_float(0x7FC00000u);  // NaN code
  } else {
    v = (e == 0u) ? (float)m * (1.0f / 512.0f) : (float)(8u + m) * pow2f((int)e - 10);
    v *= pow2f(sc - 127);
    if (b & 0x80u) v = -v;
  }
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Four E4M3 codes (bytes of w, element 0 in the low byte) times 2^(sc - 127)
// -> four bf16 (two words, element 0 in the low half of lo).
// Fast path: every code is a normal number and the scale keeps the bf16
// exponent in range; then bf16 = sign | (e + sc - 7) << 7 | m << 4 exactly.
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, int sc, uint32_t& lo, uint32_t& hi) {
  const uint32_t ex = w & 0x78787878u;
  const bool zero_exp = ((ex - 0x08080808u) & ~ex & 0x80808080u) != 0u;
  if (!zero_exp && sc >= 8 && sc <= 245) {
    const uint32_t add = (uint32_t)(sc - 7) * 0x00800080u;
    const uint32_t x0 = __byte_perm(w, 0u, 0x4140);  // byte1 << 16 | byte0
    const uint32_t x1 = __byte_perm(w, 0u, 0x4342);  // byte3 << 16 | byte2
    lo = (((x0 & 0x007F007Fu) << 4) + add) | ((x0 & 0x00800080u) << 8);
    hi = (((x1 & 0x007F007Fu) << 4) + add) | ((x1 & 0x00800080u) << 8);
  } else {
    lo = e4m3_scaled_bf16_slow(w & 0xFFu, sc) | (e4m3_scaled_bf16_slow((w >> 8) & 0xFFu, sc) << 16);
    hi = e4m3_scaled_bf16_slow((w >> 16) & 0xFFu, sc) |
         (e4m3_scaled_bf16_slow((w >> 24) & 0xFFu, sc) << 16);
  }
}

// Block shared exponent of the OCP MX rule: floor(log2 amax) - 8, clamped to
// [-127, 127]. amax must be > 0.
__device__ __forceinline__ int mx_shared_exp(float amax) {
  int sexp = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 8;
  return sexp < -127 ? -127 : (sexp > 127 ? 127 : sexp);
}

__device__ __forceinline__ uint32_t mx_encode(float v, int sexp) {
  return (uint32_t)__nv_cvt_float_to_fp8(v * pow2f(-sexp), __NV_SATFINITE, __NV_E4M3);
}

// MXFP4 (E2M1 elements, [OCP-MX] rule with emax_elem = 2): shared exponent
// floor(log2 amax) - 2, clamped to [-127, 127]. amax must be > 0.
__device__ __forceinline__ int mx4_shared_exp(float amax) {
  int sexp = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 2;
  return sexp < -127 ? -127 : (sexp > 127 ? 127 : sexp);
}

// E2M1 code (4 bits) of v / X, X = 2^sexp: round to nearest on the grid
// 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even code (mantissa bit 0),
// saturating at 6. Each midpoint comparison is against t * X, exact in fp32
// for every X >= 2^-127, so no division is rounded. The sign bit follows v.
__device__ __forceinline__ uint32_t e2m1_encode(float v, float X) {
  const float a = fabsf(v);
  const uint32_t code = (uint32_t)(a > 0.25f * X) + (uint32_t)(a >= 0.75f * X) +
                        (uint32_t)(a > 1.25f * X) + (uint32_t)(a >= 1.75f * X) +
                        (uint32_t)(a > 2.5f * X) + (uint32_t)(a >= 3.5f * X) + (uint32_t)(a > 5.0f * X);
  return code | ((__float_as_uint(v) >> 28) & 8u);
}

}  // namespace moe
