// MX element helpers (E4M3 / E2M1 elements, E8M0 block scales; OCP MX
// v1.0): the block shared exponent and element encoding of the OCP MX
// conversion rule.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace moe {

__device__ __forceinline__ float pow2f(int e) {  // exact 2^e, -127 <= e <= 127
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
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
