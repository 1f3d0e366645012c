// MXFP8 quantisation (E4M3 elements, one E8M0 scale per 32 consecutive
// elements of a row): the dynamic activation quantisation of the W8A8 MXFP8
// path ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.2:
// routed and shared Linears in MXFP8; section 六: npu_dynamic_mx_quant
// produces dynamic MXFP8 values). The rule is the OCP MX v1.0 conversion:
//   shared_exp = floor(log2(amax)) - 8   (8 = largest E4M3 exponent)
//   scale code = clamp(shared_exp, -127, 127) + 127;  amax == 0 -> code 0
//   element    = RNE(v / 2^shared_exp) to E4M3, saturating at +-448
// One thread per block of 32: 64 bytes in (four 16-byte loads), 32 code
// bytes out (two 16-byte stores) and one scale byte.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float pow2f(int e) {  // exact 2^e for -127 <= e <= 127
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

__global__ void __launch_bounds__(256) mx_quant_kernel(const uint4* __restrict__ in,
                                                       long long nblocks,
                                                       uint4* __restrict__ q,
                                                       uint8_t* __restrict__ scale) {
  const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  uint4 raw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) raw[j] = __ldg(in + b * 4 + j);
  const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(raw);
  float f[32];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    f[j] = __bfloat162float(v[j]);
    amax = fmaxf(amax, fabsf(f[j]));
  }
  uint32_t words[8];
  if (amax == 0.0f) {
    scale[b] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) words[j] = 0u;
  } else {
    const int e_amax = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;  // floor(log2 amax)
    int sexp = e_amax - 8;  // fp32-subnormal amax lands below -127 and clamps
    sexp = sexp < -127 ? -127 : (sexp > 127 ? 127 : sexp);
    scale[b] = (uint8_t)(sexp + 127);
    const float inv = pow2f(-sexp);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(f[4 * j + k] * inv, __NV_SATFINITE, __NV_E4M3);
        w |= (uint32_t)c << (8 * k);
      }
      words[j] = w;
    }
  }
  q[b * 2] = make_uint4(words[0], words[1], words[2], words[3]);
  q[b * 2 + 1] = make_uint4(words[4], words[5], words[6], words[7]);
}

}  // namespace

cudaError_t launch_mx_quantize(const void* in_bf16, int64_t rows, int cols, uint8_t* q,
                               uint8_t* scale, cudaStream_t s) {
  const long long nblocks = (long long)rows * (cols / 32);
  if (nblocks == 0) return cudaSuccess;
  const long long grid = (nblocks + 255) / 256;
  mx_quant_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint4*>(in_bf16), nblocks,
                                                 reinterpret_cast<uint4*>(q), scale);
  return cudaGetLastError();
}

}  // namespace moe
