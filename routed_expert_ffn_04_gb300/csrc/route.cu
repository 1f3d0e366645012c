// Step 1: sigmoid top-k routing with route_norm and router_scaling_factor.
// "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 一: top-8
// sigmoid routing over 192 experts; HYV3Config router_scaling_factor=2.826,
// route_norm=True, moe_router_use_sigmoid=True.
//
// One warp per token. Each lane holds ceil(E/32) logits as 64-bit keys:
//   key = (order-preserving bits of the fp32 logit) << 32 | (0xFFFFFFFF - id)
// so the largest key is the largest logit and, among equal logits, the lowest
// id. K rounds of a warp max-reduction pick the experts in slot order; the
// winning lane clears its key. Key 0 marks an empty / taken slot.
#include <cuda_runtime.h>

#include "internal.h"
#include "topk_key.cuh"

namespace moe {
namespace {

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int K, float scaling, int route_norm,
                                                    int32_t* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;

  unsigned long long key[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = j * 32 + lane;
    key[j] = (e < E) ? make_key(__ldg(row + e), e) : 0ull;
  }

  int my_id = 0;          // lane k keeps the id of slot k
  float my_logit = 0.0f;  // and its logit
  for (int k = 0; k < K; ++k) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < VPL; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, off);
      best = o > best ? o : best;
    }
    const int id = key_id(best);
    if ((id & 31) == lane) {
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (j == (id >> 5)) key[j] = 0ull;
    }
    if (lane == k) {
      my_id = id;
      my_logit = key_logit(best);
    }
  }

  // sigma(l) = 1 / (1 + exp(-l)); route_norm divides by the sum over the K slots.
  const float sig = (lane < K) ? 1.0f / (1.0f + expf(-my_logit)) : 0.0f;
  float sum = sig;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < K) {
    const float w = route_norm ? sig / sum : sig;
    topk_idx[(size_t)t * K + lane] = my_id;
    topk_w[(size_t)t * K + lane] = w * scaling;
  }
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
