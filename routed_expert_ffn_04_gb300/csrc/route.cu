// Step 1: sigmoid top-k routing with route_norm and router_scaling_factor.
// "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 一: top-8
// sigmoid routing over 192 experts; HYV3Config router_scaling_factor=2.826,
// route_norm=True, moe_router_use_sigmoid=True.
//
// One warp per token (route_warp.cuh): each lane holds ceil(E/32) logits as
// 64-bit keys, K rounds of a warp max-reduction pick the experts in slot order.
#include <cuda_runtime.h>

#include "internal.h"
#include "route_warp.cuh"

namespace moe {
namespace {

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int K, float scaling, int route_norm,
                                                    int32_t* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token_warp<VPL>(logits + (size_t)t * E, E, K, scaling, route_norm,
                        topk_idx + (size_t)t * K, topk_w + (size_t)t * K);
}

template <int VPL>
cudaError_t launch_vpl(const float* logits, int T, int E, int K, float scaling, int route_norm,
                       int32_t* idx, float* w, cudaStream_t s) {
  const int warps = 8;
  const int grid = (T + warps - 1) / warps;
  route_kernel<VPL><<<grid, warps * 32, 0, s>>>(logits, T, E, K, scaling, route_norm, idx, w);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int K, float scaling, int route_norm,
                         int32_t* topk_idx, float* topk_w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) return launch_vpl<1>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
  if (vpl <= 2) return launch_vpl<2>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
  if (vpl <= 4) return launch_vpl<4>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
  if (vpl <= 6) return launch_vpl<6>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
  if (vpl <= 8) return launch_vpl<8>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
  if (vpl <= 16) return launch_vpl<16>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
  return launch_vpl<32>(logits, T, E, K, scaling, route_norm, topk_idx, topk_w, s);
}

}  // namespace moe
