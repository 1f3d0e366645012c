// Step 2: InitRouting — stable expert-contiguous permutation of the T*K
// (token, slot) pairs and the row gather of the activations.
// "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.1 (InitRouting
// matches tokens to experts) and section 8.5 (InitRouting -> grouped GMM ->
// FinalizeRouting).
//
// Counting sort in three kernels, deterministic and without float atomics:
//   1. hist:    each warp counts expert ids over its chunk of 256 flat
//               indices (shared-memory counters) -> hist[e][w].
//   2. scan:    one block turns hist (expert-major) into exclusive bases
//               (expert totals, a scan over experts, then per-expert rows);
//               offsets[e] = base[e][0], counts[e] = the expert's total.
//   3. scatter: each warp walks its chunk in flat order, 32 at a time; lanes
//               with equal ids are grouped with __match_any_sync and ranked
//               by lane order, so rows of one expert keep ascending f.
// Up to kSmallMaxTK pairs the three run as the phases of one 1024-thread
// block (perm_small_kernel), with the per-warp counters in shared memory: the
// same counting sort, one launch instead of three.
// A fourth kernel copies each token's row to its K permuted places with
// 16-byte vector copies, reading the row once.
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr int kChunk = 256;   // flat indices per warp
constexpr int kWarps = 8;     // warps per block in hist / scatter
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kWarps * 32) perm_hist_kernel(const int32_t* __restrict__ idx,
                                                                int TK, int E, int NW,
                                                                int32_t* __restrict__ hist,
                                                                int* status) {
  extern __shared__ int32_t sh_hist[];  // [kWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarps + warp;
  int32_t* h = sh_hist + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (w >= NW) return;
  for (int p = 0; p < kChunk / 32; ++p) {
    const int f = w * kChunk + p * 32 + lane;
    if (f < TK) {
      const int e = __ldg(idx + f);
      if ((unsigned)e < (unsigned)E) atomicAdd(h + e, 1);
      else atomicCAS(status, 0, MOE_DEV_BAD_EXPERT_ID);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[(size_t)e * NW + w] = h[e];
}

// Exclusive scan of the E x NW counts in place (expert-major), by one block
// of 32 warps: (1) warp w sums the rows of experts w, w+32, ... with
// coalesced loads; (2) one exclusive scan over the E expert totals gives the
// expert offsets; (3) each warp scans its experts' rows 32 entries at a time,
// starting from the expert offset.
__global__ void __launch_bounds__(kScanThreads) perm_scan_kernel(int32_t* __restrict__ hist, int E,
                                                                 int NW, int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ offsets) {
  __shared__ int32_t tot[1024];
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = warp; e < E; e += 32) {
    const int32_t* row = hist + (size_t)e * NW;
    int32_t sum = 0;
    for (int w = lane; w < NW; w += 32) sum += row[w];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    if (lane == 0) tot[e] = sum;
  }
  __syncthreads();
  // Block exclusive scan of tot[0..E) (one entry per thread, E <= 1024).
  const int32_t v = tid < E ? tot[tid] : 0;
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t wv = warp_tot[lane];
    int32_t winc = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, winc, off);
      if (lane >= off) winc += u;
    }
    warp_tot[lane] = winc - wv;
  }
  __syncthreads();
  const int32_t excl = warp_tot[warp] + incl - v;
  if (tid < E) {
    offsets[tid] = excl;
    counts[tid] = v;
    if (tid == E - 1) offsets[E] = excl + v;
    tot[tid] = excl;  // expert start, read back below
  }
  __syncthreads();
  for (int e = warp; e < E; e += 32) {
    int32_t* row = hist + (size_t)e * NW;
    int32_t carry = tot[e];
    for (int w0 = 0; w0 < NW; w0 += 32) {
      const int w = w0 + lane;
      const int32_t c = w < NW ? row[w] : 0;
      int32_t inc = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, inc, off);
        if (lane >= off) inc += u;
      }
      if (w < NW) row[w] = carry + inc - c;
      carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32) perm_scatter_kernel(
    const int32_t* __restrict__ idx, int TK, int E, int NW, const int32_t* __restrict__ base,
    int32_t* __restrict__ perm_src, int32_t* __restrict__ flat_to_perm) {
  extern __shared__ int32_t sh_run[];  // [kWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarps + warp;
  if (w >= NW) return;
  int32_t* run = sh_run + warp * E;
  for (int e = lane; e < E; e += 32) run[e] = base[(size_t)e * NW + w];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int p = 0; p < kChunk / 32; ++p) {
    const int f = w * kChunk + p * 32 + lane;
    int e = -1;
    if (f < TK) {
      e = __ldg(idx + f);
      if ((unsigned)e >= (unsigned)E) e = -1;
    }
    const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(same & lt_mask);
    const int leader = __ffs(same) - 1;
    int pos = 0;
    if (e >= 0) pos = run[e] + rank;
    __syncwarp();
    if (e >= 0 && lane == leader) run[e] += __popc(same);
    __syncwarp();
    if (e >= 0) {
      perm_src[pos] = f;
      flat_to_perm[f] = pos;
    } else if (f < TK) {
      flat_to_perm[f] = -1;  // an invalid expert id (reported by the histogram): no row
    }
  }
}

// Counting sort of up to kSmallMaxTK pairs by one block: warp w (w < NW) owns
// flat indices [w*chunk, (w+1)*chunk). Phase 1 counts them per expert into
// hist[w][e]; phase 2 turns the counts into exclusive bases (warps in order
// within an expert, experts in order) and writes counts / offsets; phase 3
// ranks equal ids within each 32-index step with __match_any_sync, as
// perm_scatter_kernel does, so rows of one expert keep ascending f.
constexpr int kSmallMaxTK = 16384;
constexpr int kSmallThreads = 1024;
constexpr int kSmallHistInts = 12224;  // counters (NW * E <= this) + 128 B static < 48 KB

__global__ void __launch_bounds__(kSmallThreads) perm_small_kernel(
    const int32_t* __restrict__ idx, int TK, int E, int NW, int chunk,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ flat_to_perm, int* status) {
  extern __shared__ int32_t hist[];  // [NW][E]
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < NW * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();

  if (warp < NW) {
    int32_t* h = hist + warp * E;
    for (int p = 0; p < chunk; p += 32) {
      const int f = warp * chunk + p + lane;
      if (f < TK) {
        const int e = __ldg(idx + f);
        if ((unsigned)e < (unsigned)E) atomicAdd(h + e, 1);
        else atomicCAS(status, 0, MOE_DEV_BAD_EXPERT_ID);
      }
    }
  }
  __syncthreads();

  // Thread e: bases of expert e relative to its start, and its total.
  int32_t v = 0;
  if (tid < E)
    for (int w = 0; w < NW; ++w) {
      const int32_t c = hist[w * E + tid];
      hist[w * E + tid] = v;
      v += c;
    }
  // Block exclusive scan of the totals (E <= 1024 = one entry per thread).
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t wv = warp_tot[lane];
    int32_t winc = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, winc, off);
      if (lane >= off) winc += u;
    }
    warp_tot[lane] = winc - wv;
  }
  __syncthreads();
  const int32_t excl = warp_tot[warp] + incl - v;
  if (tid < E) {
    offsets[tid] = excl;
    counts[tid] = v;
    if (tid == E - 1) offsets[E] = excl + v;
    for (int w = 0; w < NW; ++w) hist[w * E + tid] += excl;
  }
  __syncthreads();

  if (warp < NW) {
    int32_t* run = hist + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int p = 0; p < chunk; p += 32) {
      const int f = warp * chunk + p + lane;
      int e = -1;
      if (f < TK) {
        e = __ldg(idx + f);
        if ((unsigned)e >= (unsigned)E) e = -1;
      }
      const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
      const int rank = __popc(same & lt_mask);
      const int leader = __ffs(same) - 1;
      int pos = 0;
      if (e >= 0) pos = run[e] + rank;
      __syncwarp();
      if (e >= 0 && lane == leader) run[e] += __popc(same);
      __syncwarp();
      if (e >= 0) {
        perm_src[pos] = f;
        flat_to_perm[f] = pos;
      } else if (f < TK) {
        flat_to_perm[f] = -1;  // an invalid expert id (reported in phase 1): no row
      }
    }
  }
}

// Work unit = (source token t, chunk of 32 x CH vectors of its row), one warp
// each, grid-stride: the chunk is read once and written to the token's K
// destination rows (flat_to_perm). Rows of x are then read from DRAM once,
// where a copy per destination row re-read them K times as the write stream
// pushed them out of L2. A pair with flat_to_perm = -1 (an invalid expert id,
// already reported) is skipped; any other index outside [0, TK) is reported.
template <typename V, int CH>
__global__ void __launch_bounds__(256) scatter_rows_kernel(const V* __restrict__ src, int T, int vecs,
                                                           const int32_t* __restrict__ flat_to_perm,
                                                           int K, int TK, V* __restrict__ dst,
                                                           int* status) {
  const int lane = threadIdx.x & 31;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const int chunks = (vecs + 32 * CH - 1) / (32 * CH);
  const long long units = (long long)T * chunks;
  for (long long u = gw; u < units; u += nw) {
    const int t = (int)(u / chunks);
    const int c0 = (int)(u - (long long)t * chunks) * 32 * CH;
    int my_p = lane < K ? __ldg(flat_to_perm + (size_t)t * K + lane) : -1;
    if (lane < K && my_p != -1 && (unsigned)my_p >= (unsigned)TK) {
      if (c0 == 0) atomicCAS(status, 0, MOE_DEV_BAD_PERM_INDEX);
      my_p = -1;
    }
    const V* s = src + (size_t)t * vecs;
    V a[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int v = c0 + j * 32 + lane;
      a[j] = v < vecs ? __ldg(s + v) : V{};
    }
    for (int k = 0; k < K; ++k) {
      const int p = __shfl_sync(0xFFFFFFFFu, my_p, k);
      if (p < 0) continue;  // warp-uniform
      V* d = dst + (size_t)p * vecs;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int v = c0 + j * 32 + lane;
        if (v < vecs) d[v] = a[j];
      }
    }
  }
}

}  // namespace

size_t permute_scratch_bytes(int TK, int E) {
  const size_t NW = (size_t)(TK + kChunk - 1) / kChunk;
  return align_up((size_t)E * (NW > 0 ? NW : 1) * sizeof(int32_t), 256);
}

cudaError_t launch_permute_index(const int32_t* topk_idx, int TK, int E, void* scratch,
                                 int32_t* counts, int32_t* offsets, int32_t* perm_src,
                                 int32_t* flat_to_perm, int* status, cudaStream_t s) {
  if (TK > 0 && TK <= kSmallMaxTK) {
    int nw = (TK + 31) / 32;
    if (nw > 32) nw = 32;
    if (nw > kSmallHistInts / E) nw = kSmallHistInts / E;
    const int chunk = ((TK + nw - 1) / nw + 31) / 32 * 32;
    perm_small_kernel<<<1, kSmallThreads, (size_t)nw * E * sizeof(int32_t), s>>>(
        topk_idx, TK, E, nw, chunk, counts, offsets, perm_src, flat_to_perm, status);
    return cudaGetLastError();
  }
  const int NW = (TK + kChunk - 1) / kChunk;
  int32_t* hist = static_cast<int32_t*>(scratch);
  const size_t smem = (size_t)kWarps * E * sizeof(int32_t);
  const int blocks = (NW + kWarps - 1) / kWarps;
  if (NW > 0) {
    perm_hist_kernel<<<blocks, kWarps * 32, smem, s>>>(topk_idx, TK, E, NW, hist, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (NW == 0) {  // no (token, slot) pairs: every expert is empty
    cudaError_t err = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    if (err == cudaSuccess) err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    return err;
  }
  perm_scan_kernel<<<1, kScanThreads, 0, s>>>(hist, E, NW, counts, offsets);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  perm_scatter_kernel<<<blocks, kWarps * 32, smem, s>>>(topk_idx, TK, E, NW, hist, perm_src,
                                                         flat_to_perm);
  return cudaGetLastError();
}

cudaError_t launch_scatter_rows(const void* src, int T, int row_bytes, const int32_t* flat_to_perm,
                                int K, int TK, void* dst, int* status, cudaStream_t s) {
  if (T == 0 || TK == 0) return cudaSuccess;
  constexpr int kCH = 4;  // 2 KB of a bf16 row per unit with 16-byte vectors
  const bool v16 = row_bytes % 16 == 0;
  const int vecs = v16 ? row_bytes / 16 : row_bytes / 4;
  const long long units = (long long)T * ((vecs + 32 * kCH - 1) / (32 * kCH));
  const long long want = (units + 7) / 8;  // 8 warps a block
  const int blocks = want < 152 * 16 ? (int)want : 152 * 16;
  if (v16) {
    scatter_rows_kernel<uint4, kCH><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), T, vecs,
                                                           flat_to_perm, K, TK,
                                                           static_cast<uint4*>(dst), status);
  } else {
    scatter_rows_kernel<uint32_t, kCH><<<blocks, 256, 0, s>>>(static_cast<const uint32_t*>(src), T,
                                                              vecs, flat_to_perm, K, TK,
                                                              static_cast<uint32_t*>(dst), status);
  }
  return cudaGetLastError();
}


}  // namespace moe
