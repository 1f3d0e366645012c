// MXFP8 quantisation (E4M3 elements, one E8M0 scale per 32 consecutive
// elements of a row): the dynamic activation quantisation of the W8A8 MXFP8
// path ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.2:
// routed and shared Linears in MXFP8; section 六: npu_dynamic_mx_quant
// produces dynamic MXFP8 values). The rule is the OCP MX v1.0 conversion:
//   shared_exp = floor(log2(amax)) - 8   (8 = largest E4M3 exponent)
//   scale code = clamp(shared_exp, -127, 127) + 127;  amax == 0 -> code 0
//   element    = RNE(v / 2^shared_exp) to E4M3, saturating at +-448
// MXFP4 (the W4A8 routed-expert weights of section 8.2) follows the same rule
// with E2M1 elements (emax_elem = 2, saturating at +-6), two codes per byte.
//
// One thread per block of 32: 64 bytes in (four 16-byte loads), 32 code
// bytes out (two 16-byte stores) and one scale byte, row-major and/or in the
// scale atoms of the block-scaled GEMM (mx_layout.cuh).
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx.cuh"
#include "mx_layout.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) mx_quant_kernel(const uint4* __restrict__ in,
                                                       long long nblocks,
                                                       uint4* __restrict__ q,
                                                       uint8_t* __restrict__ scale,
                                                       uint8_t* __restrict__ atoms, int nb) {
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
  int code = 0;
  if (amax == 0.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) words[j] = 0u;
  } else {
    const int sexp = mx_shared_exp(amax);  // an fp32-subnormal amax clamps to -127
    code = sexp + 127;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) w |= mx_encode(f[4 * j + k], sexp) << (8 * k);
      words[j] = w;
    }
  }
  if (scale) scale[b] = (uint8_t)code;
  if (atoms) {  // nb = blocks per row, a multiple of 4
    const long long row = b / nb;
    const int blk = (int)(b - row * nb);
    atoms[((row >> 7) * (nb >> 2) + (blk >> 2)) * kAtomBytes + atom_byte((int)(row & 127), blk & 3)] =
        (uint8_t)code;
  }
  if (q) {
    q[b * 2] = make_uint4(words[0], words[1], words[2], words[3]);
    q[b * 2 + 1] = make_uint4(words[4], words[5], words[6], words[7]);
  }
}

// MXFP4: one thread per block of 32 bf16 -> 16 bytes of packed E2M1 codes
// (element 2j in the low nibble) and one E8M0 scale byte.
__global__ void __launch_bounds__(256) mx4_quant_kernel(const uint4* __restrict__ in,
                                                        long long nblocks, uint4* __restrict__ q,
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
  uint32_t words[4] = {0u, 0u, 0u, 0u};
  int code = 0;
  if (amax != 0.0f) {
    const int sexp = mx4_shared_exp(amax);
    code = sexp + 127;
    const float X = pow2f(sexp);
#pragma unroll
    for (int j = 0; j < 32; ++j) words[j >> 3] |= e2m1_encode(f[j], X) << (4 * (j & 7));
  }
  scale[b] = (uint8_t)code;
  q[b] = make_uint4(words[0], words[1], words[2], words[3]);
}

}  // namespace

cudaError_t launch_mx_quantize(const void* in_bf16, int64_t rows, int cols, uint8_t* q,
                               uint8_t* scale, uint8_t* atoms, cudaStream_t s) {
  const long long nblocks = (long long)rows * (cols / 32);
  if (nblocks == 0) return cudaSuccess;
  if (atoms && cols % 128) return cudaErrorInvalidValue;
  const long long grid = (nblocks + 255) / 256;
  mx_quant_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint4*>(in_bf16), nblocks,
                                                 reinterpret_cast<uint4*>(q), scale, atoms,
                                                 cols / 32);
  return cudaGetLastError();
}

cudaError_t launch_mx4_quantize(const void* in_bf16, int64_t rows, int cols, uint8_t* q,
                                uint8_t* scale, cudaStream_t s) {
  const long long nblocks = (long long)rows * (cols / 32);
  if (nblocks == 0) return cudaSuccess;
  const long long grid = (nblocks + 255) / 256;
  mx4_quant_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint4*>(in_bf16), nblocks,
                                                  reinterpret_cast<uint4*>(q), scale);
  return cudaGetLastError();
}

}  // namespace moe
