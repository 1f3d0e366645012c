// Step 4: FinalizeRouting fused with the router scaling (already inside
// topk_w) and the shared-expert add.
// "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the main
// stream ends with the combine add. "HunyuanImage-3.0 MoE 多流变体实战",
// 源码级实现拆解 §3: output = hidden_states_mlp + combined_output.
//
//   out[t] = bf16_rne( sum_{k=0..K-1} w[t,k] * y_perm[flat_to_perm[t*K+k]] + s[t] )
//
// One block per token (grid-stride); each thread owns 4 consecutive columns
// and reads them with 16-byte loads; the sum runs over k ascending in fp32
// and is rounded to bf16 once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxK = 32;

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
        atomicCAS(status, 0, MOE_DEV_BAD_PERM_INDEX);
        p = -1;
      }
      sp[threadIdx.x] = p;
      sw[threadIdx.x] = w;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < H4; c += blockDim.x) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < K; ++k) {
        const int p = sp[k];
        if (p < 0) continue;
        const float w = sw[k];
        const float4 v = __ldg(reinterpret_cast<const float4*>(y_perm + (size_t)p * H) + c);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
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
  int grid = T < 152 * 16 ? T : 152 * 16;
  combine_kernel<<<grid, threads, 0, s>>>(y_perm, topk_w, flat_to_perm, shared_out, T, K, H,
                                          static_cast<__nv_bfloat16*>(out), status);
  return cudaGetLastError();
}

}  // namespace moe
