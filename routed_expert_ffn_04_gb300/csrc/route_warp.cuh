// Sigmoid top-k routing of one token by one warp ("腾讯混元 Hy3 在 CANN NPU 上的
// 高性能推理部署与优化实战", section 一: top-8 sigmoid routing over 192 experts;
// HYV3Config router_scaling_factor=2.826, route_norm=True).
//
// Each lane holds ceil(E/32) logits as 64-bit keys (topk_key.cuh), so the
// largest key is the largest logit and, among equal logits, the lowest id.
// K rounds of a warp max-reduction pick the experts in slot order; the
// winning lane clears its key. Lane k ends with slot k; the weights are
// sigma(logit), divided by their sum over the K slots when route_norm is set,
// times the scaling factor.
#pragma once

#include <cstdint>

#include "topk_key.cuh"

namespace moe {

// `row` holds the token's E fp32 logits (global or shared memory); called by
// all 32 lanes of a warp. Writes idx_out[0..K-1] and w_out[0..K-1].
template <int VPL>
__device__ __forceinline__ void route_token_warp(const float* row, int E, int K, float scaling,
                                                 int route_norm, int32_t* idx_out, float* w_out) {
  const int lane = threadIdx.x & 31;
  unsigned long long key[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = j * 32 + lane;
    key[j] = (e < E) ? make_key(row[e], e) : 0ull;
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
    const bool mine = (id & 31) == lane;
#pragma unroll
    for (int j = 0; j < VPL; ++j) key[j] = (mine && j == (id >> 5)) ? 0ull : key[j];
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
    idx_out[lane] = my_id;
    w_out[lane] = w * scaling;
  }
}

}  // namespace moe
