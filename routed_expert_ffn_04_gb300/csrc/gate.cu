// Steps 0+1 for few tokens: the gating projection logits[t, e] = sum_c
// x[t,c] Wr[e,c] and the sigmoid top-k routing of each token in one launch
// ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the
// gating projection, then top-k routing, is the MoE block's first stage;
// section 一: 192 experts, top-8 sigmoid routing).
//
// With few tokens the projection is a stream of the router weights (E x H
// bf16) and its arithmetic is small, so one 128-token tensor-core tile that
// walks the whole H is mostly idle SMs. Here the work is spread instead:
//   - a cluster of kCS CTAs takes TT tokens; CTA rank r takes the K range
//     [r H/kCS, (r+1) H/kCS) of every expert;
//   - inside a CTA, thread (s, e) takes expert e and the s-th of `nsplit`
//     pieces of that range, and accumulates the TT dot products in fp32 on the
//     CUDA cores, reading its weights straight from global memory (16 B a load)
//     and the tokens' x from shared memory (broadcast);
//   - partial sums are added in a fixed order: the nsplit pieces in the CTA,
//     then the kCS ranks through distributed shared memory, so the logits do
//     not depend on scheduling;
//   - rank r (r < TT) owns token r of the cluster: it reduces that token's E
//     logits over the cluster and one warp routes it (route_warp.cuh), the
//     same code as the routing kernel.
// No global scratch is used, so the result is the same whether or not the
// caller asks for the logits.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "route_warp.cuh"

namespace moe {
namespace {

namespace cg = cooperative_groups;

constexpr int kCS = 8;                    // CTAs per cluster (K pieces); portable size
constexpr int kMaxThreads = 512;
constexpr int kSmemBudget = 200 * 1024;   // dynamic shared memory a CTA may take

struct SmallGeo {
  int TT, EP, nsplit, KC;
  size_t smem;
};

SmallGeo small_geo(int T, int H, int E) {
  SmallGeo g;
  g.TT = T <= 64 ? 2 : T <= 128 ? 4 : 8;  // about 32 clusters from 64 tokens up
  g.EP = (E + 31) / 32 * 32;
  g.KC = H / kCS;
  g.nsplit = 1;
  for (int n = 4; n >= 2; n >>= 1)
    if (n * g.EP <= kMaxThreads && g.KC % (8 * n) == 0) {
      g.nsplit = n;
      break;
    }
  g.smem = ((size_t)g.TT * g.KC + (size_t)g.nsplit * g.TT * g.EP + g.EP) * sizeof(float);
  return g;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float* f) {
  const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(u[j] << 16);
    f[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
  }
}

// Shared memory: xs [TT][KC] fp32 | part [nsplit][TT][EP] fp32 | lg [EP] fp32.
template <int TT, int VPL>
__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kMaxThreads)
    gate_route_small_kernel(const __nv_bfloat16* __restrict__ x,
                            const __nv_bfloat16* __restrict__ wr, int T, int H, int E, int K,
                            float scaling, int route_norm, int nsplit,
                            float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                            float* __restrict__ topk_w) {
  extern __shared__ __align__(16) float smem[];
  cg::cluster_group cl = cg::this_cluster();
  const int r = (int)cl.block_rank();
  const int t0 = (blockIdx.x / kCS) * TT;
  const int EP = (E + 31) / 32 * 32;
  const int KC = H / kCS;
  const int KS = KC / nsplit;
  const int k0 = r * KC;
  float* xs = smem;
  float* part = xs + TT * KC;
  float* lg = part + nsplit * TT * EP;

  // x[t0 .. t0+TT-1, k0 .. k0+KC-1] -> fp32 (rows past T are zero).
  const int vec_per_row = KC / 8;
  for (int i = threadIdx.x; i < TT * vec_per_row; i += blockDim.x) {
    const int t = i / vec_per_row, c = i - t * vec_per_row;
    float f[8];
    if (t0 + t < T) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * H + k0) + c);
      bf16x8_to_f32(q, f);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = 0.0f;
    }
    float4* d = reinterpret_cast<float4*>(xs + t * KC + 8 * c);
    d[0] = make_float4(f[0], f[1], f[2], f[3]);
    d[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  __syncthreads();

  const int s = threadIdx.x / EP, e = threadIdx.x - s * EP;
  float a0[TT], a1[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) a0[t] = a1[t] = 0.0f;
  if (e < E) {
    const uint4* wp = reinterpret_cast<const uint4*>(wr + (size_t)e * H + k0 + s * KS);
    const float* xp = xs + s * KS;
#pragma unroll 4
    for (int v = 0; v < KS / 8; ++v) {
      float wf[8];
      bf16x8_to_f32(__ldg(wp + v), wf);
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const float4 xa = *reinterpret_cast<const float4*>(xp + t * KC + 8 * v);
        const float4 xb = *reinterpret_cast<const float4*>(xp + t * KC + 8 * v + 4);
        a0[t] = fmaf(xa.x, wf[0], a0[t]);
        a1[t] = fmaf(xa.y, wf[1], a1[t]);
        a0[t] = fmaf(xa.z, wf[2], a0[t]);
        a1[t] = fmaf(xa.w, wf[3], a1[t]);
        a0[t] = fmaf(xb.x, wf[4], a0[t]);
        a1[t] = fmaf(xb.y, wf[5], a1[t]);
        a0[t] = fmaf(xb.z, wf[6], a0[t]);
        a1[t] = fmaf(xb.w, wf[7], a1[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TT; ++t) part[(s * TT + t) * EP + e] = a0[t] + a1[t];
  __syncthreads();
  // The nsplit pieces of this CTA, in order, into piece 0.
  for (int i = threadIdx.x; i < TT * EP; i += blockDim.x) {
    float v = part[i];
    for (int q = 1; q < nsplit; ++q) v += part[q * TT * EP + i];
    part[i] = v;
  }
  cl.sync();  // every rank's partial logits are complete

  const bool owner = r < TT && t0 + r < T;
  if (owner && threadIdx.x < E) {
    float v = 0.0f;
#pragma unroll
    for (int q = 0; q < kCS; ++q) v += cl.map_shared_rank(part, q)[r * EP + threadIdx.x];
    lg[threadIdx.x] = v;
    if (logits) logits[(size_t)(t0 + r) * E + threadIdx.x] = v;
  }
  cl.sync();  // no rank leaves while another still reads its partials

  if (owner && threadIdx.x < 32)
    route_token_warp<VPL>(lg, E, K, scaling, route_norm, topk_idx + (size_t)(t0 + r) * K,
                          topk_w + (size_t)(t0 + r) * K);
}

template <int TT, int VPL>
cudaError_t launch_tt(const __nv_bfloat16* x, const __nv_bfloat16* wr, int T, int H, int E,
                      int K, float scaling, int route_norm, const SmallGeo& g, float* logits,
                      int32_t* idx, float* w, cudaStream_t s) {
  const int clusters = (T + TT - 1) / TT;
  gate_route_small_kernel<TT, VPL><<<clusters * kCS, g.nsplit * g.EP, g.smem, s>>>(
      x, wr, T, H, E, K, scaling, route_norm, g.nsplit, logits, idx, w);
  return cudaGetLastError();
}

template <int TT>
cudaError_t set_smem_limits() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(gate_route_small_kernel<TT, 1>, a, kSmemBudget);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gate_route_small_kernel<TT, 2>, a, kSmemBudget);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gate_route_small_kernel<TT, 4>, a, kSmemBudget);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gate_route_small_kernel<TT, 8>, a, kSmemBudget);
  return e;
}

template <int VPL>
cudaError_t launch_vpl(const __nv_bfloat16* x, const __nv_bfloat16* wr, int T, int H, int E,
                       int K, float scaling, int route_norm, const SmallGeo& g, float* logits,
                       int32_t* idx, float* w, cudaStream_t s) {
  switch (g.TT) {
    case 2: return launch_tt<2, VPL>(x, wr, T, H, E, K, scaling, route_norm, g, logits, idx, w, s);
    case 4: return launch_tt<4, VPL>(x, wr, T, H, E, K, scaling, route_norm, g, logits, idx, w, s);
    default: return launch_tt<8, VPL>(x, wr, T, H, E, K, scaling, route_norm, g, logits, idx, w, s);
  }
}

}  // namespace

// Shared-memory limits of every instantiation, set once per device when a
// handle is created, so that a launch makes no attribute call (graph capture).
cudaError_t gate_small_prepare_device() {
  cudaError_t e = set_smem_limits<2>();
  if (e == cudaSuccess) e = set_smem_limits<4>();
  if (e == cudaSuccess) e = set_smem_limits<8>();
  return e;
}

bool gate_route_small_fits(int T, int H, int E) {
  if (T <= 0 || T > kGateSmallMaxT || E > 256 || H % (8 * kCS)) return false;
  return small_geo(T, H, E).smem <= (size_t)kSmemBudget;
}

cudaError_t launch_gate_route_small(const void* x, const void* w_router, int T, int H, int E,
                                    int K, float scaling, int route_norm, float* logits,
                                    int32_t* topk_idx, float* topk_w, cudaStream_t s) {
  if (!gate_route_small_fits(T, H, E)) return cudaErrorInvalidValue;
  const SmallGeo g = small_geo(T, H, E);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  const auto* wb = static_cast<const __nv_bfloat16*>(w_router);
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) return launch_vpl<1>(xb, wb, T, H, E, K, scaling, route_norm, g, logits, topk_idx, topk_w, s);
  if (vpl <= 2) return launch_vpl<2>(xb, wb, T, H, E, K, scaling, route_norm, g, logits, topk_idx, topk_w, s);
  if (vpl <= 4) return launch_vpl<4>(xb, wb, T, H, E, K, scaling, route_norm, g, logits, topk_idx, topk_w, s);
  return launch_vpl<8>(xb, wb, T, H, E, K, scaling, route_norm, g, logits, topk_idx, topk_w, s);
}

}  // namespace moe
