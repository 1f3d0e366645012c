// Tile scheduling and pipeline bookkeeping shared by the grouped GEMM
// kernels (gemm.cu, gemm_mx.cu): kernel parameters, the per-group tile
// decode, ring positions and the drain helpers used when a CTA aborts.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace moe {

struct KParams {
  const int32_t* offsets;  // [G+1] or nullptr
  int G;
  int rows;
  int num_kb;    // ceil(Kdim / 64)
  int N;         // output columns per group (I for MODE 0, H for MODE 1)
  void* out;     // bf16 h (MODE 0) or fp32 y (MODE 1)
  int* status;
  uint64_t limit_ns;
  // MXFP8 (gemm_mx.cu): scale atoms of the weights, of the activations (one
  // atom row-block per token tile), and for GEMM-1 of the E4M3 h it writes.
  const uint8_t* s_w0;
  const uint8_t* s_act;
  uint8_t* out_scale;
  // Group that takes the second weight maps (a folded shared expert), or -1.
  int fold_group;
  // GEMM-1 with the row gather in its A load: row r of group g is token
  // gather_src[r] / gather_k of gather_x ([T, H] bf16); nullptr: a is given.
  const int32_t* gather_src;
  int gather_k;
  const void* gather_x;
  // Gating (MODE 2): routing outputs [rows, topk]; `out` (nullable) takes the logits.
  int32_t* topk_idx;
  float* topk_w;
  int topk;
  float scaling;
  int route_norm;
};

struct TileInfo {
  int g, row0, nrows, wt, tt;
};

// Group rows [row0, row0 + nrows), clamped to [0, rows).
__device__ __forceinline__ void group_rows(const KParams& p, int g, int& row0, int& nrows) {
  if (p.offsets == nullptr) {
    row0 = 0;
    nrows = p.rows;
    return;
  }
  int a = __ldg(p.offsets + g), b = __ldg(p.offsets + g + 1);
  a = a < 0 ? 0 : (a > p.rows ? p.rows : a);
  b = b < a ? a : (b > p.rows ? p.rows : b);
  row0 = a;
  nrows = b - a;
}

template <int ACT_ROWS>
__device__ __forceinline__ TileInfo decode_tile(const KParams& p, const int32_t* tile_start,
                                                int tile) {
  int lo = 0, hi = p.G;  // tile_start[lo] <= tile < tile_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  TileInfo t;
  t.g = lo;
  group_rows(p, lo, t.row0, t.nrows);
  const int n_tt = (t.nrows + ACT_ROWS - 1) / ACT_ROWS;
  const int local = tile - tile_start[lo];
  t.wt = local / n_tt;
  t.tt = local - t.wt * n_tt;
  return t;
}

// The same decode from a shared-memory copy of the group starts
// (row_start[g] = offsets[g] clamped to [0, rows], g = 0..G; see
// fill_row_start), so that a role starting a tile does not wait on a global
// load of the offsets.
template <int ACT_ROWS>
__device__ __forceinline__ TileInfo decode_tile_s(int G, const int32_t* tile_start,
                                                  const int32_t* row_start, int tile) {
  int lo = 0, hi = G;  // tile_start[lo] <= tile < tile_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid;
  }
  TileInfo t;
  t.g = lo;
  t.row0 = row_start[lo];
  const int nr = row_start[lo + 1] - t.row0;
  t.nrows = nr > 0 ? nr : 0;
  const int n_tt = (t.nrows + ACT_ROWS - 1) / ACT_ROWS;
  const int local = tile - tile_start[lo];
  t.wt = local / n_tt;
  t.tt = local - t.wt * n_tt;
  return t;
}

// row_start[g] for g = 0..G (executed by all `nthreads` threads of the CTA
// before a __syncthreads): rows [row_start[g], row_start[g+1]) are group g,
// as group_rows clamps them.
__device__ __forceinline__ void fill_row_start(const KParams& p, int32_t* row_start, int tid, int nthreads) {
  for (int g = tid; g <= p.G; g += nthreads) {
    int v = p.offsets ? __ldg(p.offsets + g) : (g == 0 ? 0 : p.rows);
    row_start[g] = v < 0 ? 0 : (v > p.rows ? p.rows : v);
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// Bounded wait that ignores the abort flag, used only to drain in-flight work.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) break;
  }
}

// Generic-proxy shared-memory writes become visible to the async proxy
// (tcgen05.mma operand reads) after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// A simple ring position: stage index and the parity of its current phase.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Issued-but-unobserved TMA copies per ring, drained before an aborting CTA exits.
struct Armed {
  uint32_t mask = 0, phase = 0;
  __device__ __forceinline__ void mark(const Ring& r) {
    mask |= 1u << r.s;
    phase = (phase & ~(1u << r.s)) | (r.ph << r.s);
  }
};

}  // namespace moe
