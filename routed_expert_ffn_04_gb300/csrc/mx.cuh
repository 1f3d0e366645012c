// MXFP8 element helpers (E4M3 elements, E8M0 block scales; OCP MX v1.0):
// exact expansion of scaled E4M3 codes into bf16, and the quantise ->
// dequantise round trip of the OCP MX conversion rule.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// Sixteen E4M3 codes (one 16-byte chunk) times 2^(sc - 127) -> sixteen bf16,
// stored as two 16-byte vectors at d0 (elements 0-7) and d1 (elements 8-15).
// The exact-but-slow per-code path is kept out of line; it only runs for
// chunks holding zero/subnormal codes or extreme scales.
static __device__ __noinline__ void e4m3x16_to_bf16_slow(uint4 c, int sc, uint4* d0, uint4* d1) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[8];
  for (int k = 0; k < 4; ++k)
    for (int b = 0; b < 4; b += 2)
      o[2 * k + b / 2] = e4m3_scaled_bf16_slow((w[k] >> (8 * b)) & 0xFFu, sc) |
                         (e4m3_scaled_bf16_slow((w[k] >> (8 * b + 8)) & 0xFFu, sc) << 16);
  *d0 = make_uint4(o[0], o[1], o[2], o[3]);
  *d1 = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void e4m3x16_to_bf16_store(uint4 c, int sc, uint4* d0, uint4* d1) {
  const uint32_t e0 = c.x & 0x78787878u, e1 = c.y & 0x78787878u, e2 = c.z & 0x78787878u,
                 e3 = c.w & 0x78787878u;
  const uint32_t z = ((e0 - 0x08080808u) & ~e0) | ((e1 - 0x08080808u) & ~e1) |
                     ((e2 - 0x08080808u) & ~e2) | ((e3 - 0x08080808u) & ~e3);
  if ((z & 0x80808080u) == 0u && sc >= 8 && sc <= 245) {
    const uint32_t add = (uint32_t)(sc - 7) * 0x00800080u;
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t x0 = __byte_perm(w[k], 0u, 0x4140), x1 = __byte_perm(w[k], 0u, 0x4342);
      o[2 * k] = (((x0 & 0x007F007Fu) << 4) + add) | ((x0 & 0x00800080u) << 8);
      o[2 * k + 1] = (((x1 & 0x007F007Fu) << 4) + add) | ((x1 & 0x00800080u) << 8);
    }
    *d0 = make_uint4(o[0], o[1], o[2], o[3]);
    *d1 = make_uint4(o[4], o[5], o[6], o[7]);
  } else {
    e4m3x16_to_bf16_slow(c, sc, d0, d1);
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

// Quantise v (in a block whose amax is given) to E4M3 and return the
// dequantised value (exact in bf16). amax == 0 gives +0.
__device__ __forceinline__ float mx_roundtrip(float v, float amax) {
  if (amax == 0.0f) return 0.0f;
  const int sexp = mx_shared_exp(amax);
  const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)mx_encode(v, sexp), __NV_E4M3);
  return __half2float(__half(hr)) * pow2f(sexp);
}

}  // namespace moe
