// Ordering keys of the sigmoid top-k routing ("腾讯混元 Hy3 在 CANN NPU 上的高性能
// 推理部署与优化实战", section 一): experts ranked by fp32 logit, equal logits ->
// lower expert id first, +0 equal to -0, NaN below every number.
//   key = (order-preserving bits of the logit) << 32 | (0xFFFFFFFF - id)
// so a larger key is a better expert. Key 0 marks an empty slot.
#pragma once

#include <cstdint>

namespace moe {

__device__ __forceinline__ unsigned long long make_key(float l, int id) {
  uint32_t ord;
  if (l != l) {
    ord = 0;  // NaN ranks below every number
  } else {
    l = l + 0.0f;  // -0 -> +0 so that the two zeros tie
    const uint32_t u = __float_as_uint(l);
    ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

__device__ __forceinline__ float key_logit(unsigned long long key) {
  const uint32_t ord = (uint32_t)(key >> 32);
  const uint32_t u = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(u);
}

__device__ __forceinline__ int key_id(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

}  // namespace moe
