// Step 4: FinalizeRouting fused with the router scaling (already inside
// topk_w) and the shared-expert add.
// "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the main
// stream ends with the combine add. "HunyuanImage-3.0 MoE 多流变体实战",
// 源码级实现拆解 §3: output = hidden_states_mlp + combined_output.
//
//   out[t] = bf16_rne( sum_{k=0..K-1} w[t,k] * y_perm[flat_to_perm[t*K+k]] + s[t] )
//
// Two forms with the same arithmetic (sum over k ascending in fp32, one
// bf16 rounding), chosen by the token count:
//   - many tokens: one block per token (grid-stride), each thread owns 4
//     consecutive columns at a time and reads them with 16-byte loads;
//   - few tokens (fewer than two blocks per SM): a work unit is (token, chunk
//     of 4 * blockDim columns), so that the few tokens still fill the grid.
// Both load the K rows' vectors of a column chunk in batches of 8 before
// adding them, so each thread has several loads in flight.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxK = 32;
constexpr int kSms = 152;  // grid sizing
constexpr int kBatch = 8;  // row loads in flight per thread

// out[t, 4c .. 4c+3] from the token's K rows (sp: permuted row or -1, sw:
// weight) and its shared-expert row.
__device__ __forceinline__ void combine_chunk(const float* __restrict__ y_perm,
                                              const float* __restrict__ shared_out, const float* sw,
                                              const int32_t* sp, int t, int K, int H, int c,
                                              __nv_bfloat16* __restrict__ out) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < K; k0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int p = (k0 + j < K) ? sp[k0 + j] : -1;
      v[j] = p >= 0 ? __ldg(reinterpret_cast<const float4*>(y_perm + (size_t)p * H) + c)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (k0 + j >= K || sp[k0 + j] < 0) continue;
      const float w = sw[k0 + j];
      acc.x = fmaf(w, v[j].x, acc.x);
      acc.y = fmaf(w, v[j].y, acc.y);
      acc.z = fmaf(w, v[j].z, acc.z);
      acc.w = fmaf(w, v[j].w, acc.w);
    }
  }
  if (shared_out) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(shared_out + (size_t)t * H) + c);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + (size_t)t * H)[c] = pk;
}

__global__ void __launch_bounds__(256) combine_split_kernel(const float* __restrict__ y_perm,
                                                      const float* __restrict__ topk_w,
                                                      const int32_t* __restrict__ flat_to_perm,
                                                      const float* __restrict__ shared_out, int T,
                                                      int K, int H, __nv_bfloat16* __restrict__ out,
                                                      int* status) {
  __shared__ float sw[kMaxK];
  __shared__ int32_t sp[kMaxK];
  const int TK = T * K;
  const int H4 = H >> 2;
  const int chunks = (H4 + blockDim.x - 1) / blockDim.x;
  const long long units = (long long)T * chunks;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const int t = (int)(u / chunks);
    const int c = (int)(u - (long long)t * chunks) * blockDim.x + threadIdx.x;
    __syncthreads();
    if (threadIdx.x < K) {
      int32_t p = flat_to_perm[(size_t)t * K + threadIdx.x];
      float w = topk_w[(size_t)t * K + threadIdx.x];
      if ((unsigned)p >= (unsigned)TK) {
        // -1 marks a pair the permutation dropped (an expert id out of
        // range, already reported there): it adds nothing, silently.
        if (p != -1) atomicCAS(status, 0, MOE_DEV_BAD_PERM_INDEX);
        p = -1;
      }
      sp[threadIdx.x] = p;
      sw[threadIdx.x] = w;
    }
    __syncthreads();
    if (c >= H4) continue;
    combine_chunk(y_perm, shared_out, sw, sp, t, K, H, c, out);
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_perm,
                                                      const float* __restrict__ topk_w,
                                                      const int32_t* __restrict__ flat_to_perm,
                                                      const float* __restrict__ shared_out, int T,
                                                      int K, int H, __nv_bfloat16* __restrict__ out,
                                                      int* status) {
  __shared__ float sw[kMaxK];
  __shared__ int32_t sp[kMaxK];
  const int TK = T * K;
  const int H4 = H >> 2;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < K) {
      int32_t p = flat_to_perm[(size_t)t * K + threadIdx.x];
      float w = topk_w[(size_t)t * K + threadIdx.x];
      if ((unsigned)p >= (unsigned)TK) {
        // -1 marks a pair the permutation dropped (an expert id out of
        // range, already reported there): it adds nothing, silently.
        if (p != -1) atomicCAS(status, 0, MOE_DEV_BAD_PERM_INDEX);
        p = -1;
      }
      sp[threadIdx.x] = p;
      sw[threadIdx.x] = w;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < H4; c += blockDim.x) combine_chunk(y_perm, shared_out, sw, sp, t, K, H, c, out);
  }
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const float* topk_w, const int32_t* flat_to_perm,
                           const float* shared_out, int T, int K, int H, void* out, int* status,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  int threads = H / 4;
  if (threads > 256) threads = 256;
  threads = (threads + 31) / 32 * 32;
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (T >= 2 * kSms) {
    const int grid = T < kSms * 16 ? T : kSms * 16;
    combine_kernel<<<grid, threads, 0, s>>>(y_perm, topk_w, flat_to_perm, shared_out, T, K, H, o,
                                            status);
  } else {
    const long long units = (long long)T * ((H / 4 + threads - 1) / threads);
    const int grid = units < kSms * 16 ? (int)units : kSms * 16;
    combine_split_kernel<<<grid, threads, 0, s>>>(y_perm, topk_w, flat_to_perm, shared_out, T, K,
                                                  H, o, status);
  }
  return cudaGetLastError();
}

}  // namespace moe
