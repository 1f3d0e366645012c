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
// The same counting sort also runs as the phases of one launch with the
// per-warp counters in shared memory: up to kSmallMaxTK pairs in one
// 1024-thread block (perm_small_kernel), and up to kClusterMaxTK pairs in a
// cluster of 8 such blocks (perm_cluster_kernel: the blocks' per-expert
// totals are exchanged through distributed shared memory between the count
// and scatter phases). The three kernels take larger inputs.
// Each path can also write tile_offsets[e], the first 128-row tile of expert
// e (an exclusive scan of ceil(count / 128)), which is where the MX GEMMs find
// the scale atoms of an expert's rows.
// A fourth kernel copies each token's row to its K permuted places with
// 16-byte vector copies, reading the row once; in the MX layer it also
// writes each row's E8M0 scales into the scale atoms.
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "internal.h"
#include "mx_layout.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = 256;   // flat indices per warp
constexpr int kWarps = 8;     // warps per block in hist / scatter
constexpr int kScanThreads = 1024;

// Exclusive scan of one value per thread over a block of up to 1024 threads
// (warp_tot: 33 ints of shared memory). Returns the prefix; *total = the sum.
// Every thread of the block calls it.
__device__ __forceinline__ int32_t block_excl_scan(int32_t v, int32_t* warp_tot, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += u;
  }
  __syncthreads();  // warp_tot may still be read after a previous call
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    const int32_t wv = lane < nw ? warp_tot[lane] : 0;
    int32_t winc = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, winc, off);
      if (lane >= off) winc += u;
    }
    warp_tot[lane] = winc - wv;
    if (lane == 31) warp_tot[32] = winc;
  }
  __syncthreads();
  *total = warp_tot[32];
  return warp_tot[warp] + incl - v;
}

// tile_offsets[e] = sum over g < e of ceil(count_g / 128), tile_offsets[E] =
// the total; v = the count of expert threadIdx.x (0 past E). Every thread of
// the block calls it.
__device__ __forceinline__ void write_tile_offsets(int32_t v, int E, int32_t* warp_tot,
                                                   int32_t* __restrict__ tile_offsets) {
  int32_t total;
  const int32_t t = block_excl_scan((v + 127) >> 7, warp_tot, &total);
  if (threadIdx.x < E) {
    tile_offsets[threadIdx.x] = t;
    if (threadIdx.x == E - 1) tile_offsets[E] = total;
  }
}

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
                                                                 int32_t* __restrict__ offsets,
                                                                 int32_t* __restrict__ tile_offsets) {
  __shared__ int32_t tot[1024];
  __shared__ int32_t warp_tot[33];
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
  int32_t total;
  const int32_t excl = block_excl_scan(v, warp_tot, &total);
  if (tid < E) {
    offsets[tid] = excl;
    counts[tid] = v;
    if (tid == E - 1) offsets[E] = excl + v;
    tot[tid] = excl;  // expert start, read back below
  }
  if (tile_offsets) write_tile_offsets(v, E, warp_tot, tile_offsets);
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

// One warp counts the expert ids of flat indices [f0, f0 + len) (len a
// multiple of 32) into h[0..E) with shared-memory atomics; an id outside
// [0, E) is reported in the status word.
__device__ __forceinline__ void count_chunk(const int32_t* __restrict__ idx, int TK, int E, int f0,
                                            int len, int32_t* h, int* status) {
  const int lane = threadIdx.x & 31;
  for (int p = 0; p < len; p += 32) {
    const int f = f0 + p + lane;
    if (f < TK) {
      const int e = __ldg(idx + f);
      if ((unsigned)e < (unsigned)E) atomicAdd(h + e, 1);
      else atomicCAS(status, 0, MOE_DEV_BAD_EXPERT_ID);
    }
  }
}

// One warp places the flat indices [f0, f0 + len) in flat order: run[e] is
// the next permuted row of expert e for this warp. Within each step of 32,
// lanes with equal ids are grouped with __match_any_sync and ranked by lane,
// so the rows of one expert keep ascending f.
__device__ __forceinline__ void scatter_chunk(const int32_t* __restrict__ idx, int TK, int E, int f0,
                                              int len, int32_t* run, int32_t* __restrict__ perm_src,
                                              int32_t* __restrict__ flat_to_perm) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int p = 0; p < len; p += 32) {
    const int f = f0 + p + lane;
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
      flat_to_perm[f] = -1;  // an invalid expert id (reported when counting): no row
    }
  }
}

// Counting sort of up to kSmallMaxTK pairs by one block: warp w (w < NW) owns
// flat indices [w*chunk, (w+1)*chunk). Phase 1 counts them per expert into
// hist[w][e]; phase 2 turns the counts into exclusive bases (warps in order
// within an expert, experts in order) and writes counts / offsets (and the
// tile offsets); phase 3 places each warp's indices (scatter_chunk).
constexpr int kSmallMaxTK = 4096;
constexpr int kSmallThreads = 1024;
constexpr int kSmallHistInts = 12224;  // counters (NW * E <= this) + static < 48 KB

__global__ void __launch_bounds__(kSmallThreads) perm_small_kernel(
    const int32_t* __restrict__ idx, int TK, int E, int NW, int chunk,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ tile_offsets,
    int32_t* __restrict__ perm_src, int32_t* __restrict__ flat_to_perm, int* status) {
  extern __shared__ int32_t hist[];  // [NW][E]
  __shared__ int32_t warp_tot[33];
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < NW * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  if (warp < NW) count_chunk(idx, TK, E, warp * chunk, chunk, hist + warp * E, status);
  __syncthreads();

  // Thread e: bases of expert e relative to its start, and its total.
  int32_t v = 0;
  if (tid < E)
    for (int w = 0; w < NW; ++w) {
      const int32_t c = hist[w * E + tid];
      hist[w * E + tid] = v;
      v += c;
    }
  int32_t total;
  const int32_t excl = block_excl_scan(v, warp_tot, &total);  // E <= 1024 = one entry per thread
  if (tid < E) {
    offsets[tid] = excl;
    counts[tid] = v;
    if (tid == E - 1) offsets[E] = excl + v;
    for (int w = 0; w < NW; ++w) hist[w * E + tid] += excl;
  }
  if (tile_offsets) write_tile_offsets(v, E, warp_tot, tile_offsets);
  __syncthreads();
  if (warp < NW) scatter_chunk(idx, TK, E, warp * chunk, chunk, hist + warp * E, perm_src, flat_to_perm);
}

// The same counting sort by a cluster of kClusterCtas blocks of 32 warps:
// warp w of CTA r owns flat indices [(32 r + w) chunk, (32 r + w + 1) chunk).
// Each CTA counts and bases its warps' indices as perm_small_kernel does,
// relative to the CTA; the CTAs' per-expert totals are then read through
// distributed shared memory, so each CTA adds the totals of the CTAs before
// it and the expert offsets (the same scan in every CTA; CTA 0 writes
// counts, offsets and tile offsets). A second cluster barrier keeps every CTA
// until all have read the others' totals.
constexpr int kClusterCtas = 8;
constexpr int kClusterThreads = 1024;
constexpr int kClusterWarps = kClusterThreads / 32;
constexpr int kClusterMaxTK = kClusterCtas * kClusterWarps * 1024;  // chunk <= 1024 per warp

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kClusterThreads)
    perm_cluster_kernel(const int32_t* __restrict__ idx, int TK, int E, int chunk,
                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ tile_offsets, int32_t* __restrict__ perm_src,
                        int32_t* __restrict__ flat_to_perm, int* status) {
  extern __shared__ int32_t hist[];  // [32][E], then this CTA's totals [E]
  int32_t* ctot = hist + kClusterWarps * E;
  __shared__ int32_t warp_tot[33];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  for (int i = tid; i < kClusterWarps * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int f0 = ((int)rank * kClusterWarps + warp) * chunk;
  count_chunk(idx, TK, E, f0, chunk, hist + warp * E, status);
  __syncthreads();

  int32_t v = 0;  // this CTA's count of expert tid (E <= 1024 = one expert per thread)
  if (tid < E) {
    for (int w = 0; w < kClusterWarps; ++w) {
      const int32_t c = hist[w * E + tid];
      hist[w * E + tid] = v;
      v += c;
    }
    ctot[tid] = v;
  }
  cluster_sync_all();
  int32_t cbase = 0, tot = 0;  // counts of the CTAs before this one; of all CTAs
  if (tid < E) {
    const uint32_t a = smem_u32(ctot + tid);
#pragma unroll
    for (int r = 0; r < kClusterCtas; ++r) {
      const int32_t c = ld_shared_cluster_s32(mapa_shared(a, (uint32_t)r));
      cbase += r < (int)rank ? c : 0;
      tot += c;
    }
  }
  int32_t total;
  const int32_t excl = block_excl_scan(tot, warp_tot, &total);
  if (tid < E) {
    if (rank == 0) {
      offsets[tid] = excl;
      counts[tid] = tot;
      if (tid == E - 1) offsets[E] = excl + tot;
    }
    for (int w = 0; w < kClusterWarps; ++w) hist[w * E + tid] += excl + cbase;
  }
  if (tile_offsets && rank == 0) write_tile_offsets(tot, E, warp_tot, tile_offsets);
  cluster_sync_all();
  scatter_chunk(idx, TK, E, f0, chunk, hist + warp * E, perm_src, flat_to_perm);
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

// MX layer: each token's E4M3 row (as scatter_rows_kernel, 16-byte vectors,
// 4 per lane per unit) and its E8M0 scales. The unit holding the start of a
// row also places the token's nk = H/128 scale words (four scales each) into
// the scale atoms the MX GEMM reads: for each of its K rows p (expert e, row
// j = p - offsets[e] of the expert), word ka goes to atom (tile_offsets[e] +
// j / 128, ka) at the position of row j % 128 (mx_layout.cuh).
__global__ void __launch_bounds__(256) scatter_rows_mx_kernel(
    const uint4* __restrict__ src, const uint32_t* __restrict__ scale_words, int T, int vecs, int nk,
    const int32_t* __restrict__ flat_to_perm, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_offsets, int K, int TK,
    int E, uint4* __restrict__ dst, uint32_t* __restrict__ atoms, int* status) {
  constexpr int CH = 4;
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
    const uint4* s = src + (size_t)t * vecs;
    uint4 a[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int v = c0 + j * 32 + lane;
      a[j] = v < vecs ? __ldg(s + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    for (int k = 0; k < K; ++k) {
      const int p = __shfl_sync(0xFFFFFFFFu, my_p, k);
      if (p < 0) continue;  // warp-uniform
      uint4* d = dst + (size_t)p * vecs;
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int v = c0 + j * 32 + lane;
        if (v < vecs) d[v] = a[j];
      }
    }
    if (c0 != 0) continue;  // warp-uniform
    // Row j of its expert and the atom row-block, per slot (lane k).
    int my_j = -1, my_blk = 0;
    if (lane < K && my_p >= 0) {
      const int e = __ldg(topk_idx + (size_t)t * K + lane);
      if ((unsigned)e < (unsigned)E) {
        my_j = my_p - __ldg(offsets + e);
        my_blk = __ldg(tile_offsets + e) + (my_j >> 7);
      }
    }
    for (int k = 0; k < K; ++k) {
      const int j = __shfl_sync(0xFFFFFFFFu, my_j, k);
      const int blk = __shfl_sync(0xFFFFFFFFu, my_blk, k);
      if (j < 0) continue;  // warp-uniform
      const int r = j & 127;
      const size_t in_atom = (size_t)(4 * (r & 31) + (r >> 5));  // atom_byte(r, 0) / 4
      for (int ka = lane; ka < nk; ka += 32)
        atoms[((size_t)blk * nk + ka) * (kAtomBytes / 4) + in_atom] = __ldg(scale_words + (size_t)t * nk + ka);
    }
  }
}

}  // namespace

size_t permute_scratch_bytes(int TK, int E) {
  const size_t NW = (size_t)(TK + kChunk - 1) / kChunk;
  return align_up((size_t)E * (NW > 0 ? NW : 1) * sizeof(int32_t), 256);
}

// Dynamic shared memory of the cluster permutation: hist [32][E] and the
// CTA's totals [E].
constexpr int kClusterSmemInts = kClusterWarps + 1;

cudaError_t permute_prepare_device() {
  return cudaFuncSetAttribute(perm_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kClusterSmemInts * 1024 * (int)sizeof(int32_t));
}

cudaError_t launch_permute_index(const int32_t* topk_idx, int TK, int E, void* scratch,
                                 int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                                 int32_t* perm_src, int32_t* flat_to_perm, int* status,
                                 cudaStream_t s) {
  if (TK > 0 && TK <= kSmallMaxTK) {
    int nw = (TK + 31) / 32;
    if (nw > 32) nw = 32;
    if (nw > kSmallHistInts / E) nw = kSmallHistInts / E;
    const int chunk = ((TK + nw - 1) / nw + 31) / 32 * 32;
    perm_small_kernel<<<1, kSmallThreads, (size_t)nw * E * sizeof(int32_t), s>>>(
        topk_idx, TK, E, nw, chunk, counts, offsets, tile_offsets, perm_src, flat_to_perm, status);
    return cudaGetLastError();
  }
  if (TK > kSmallMaxTK && TK <= kClusterMaxTK) {
    const int nwarps = kClusterCtas * kClusterWarps;
    const int chunk = ((TK + nwarps - 1) / nwarps + 31) / 32 * 32;
    perm_cluster_kernel<<<kClusterCtas, kClusterThreads, (size_t)kClusterSmemInts * E * sizeof(int32_t), s>>>(
        topk_idx, TK, E, chunk, counts, offsets, tile_offsets, perm_src, flat_to_perm, status);
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
    if (err == cudaSuccess && tile_offsets)
      err = cudaMemsetAsync(tile_offsets, 0, sizeof(int32_t) * (E + 1), s);
    return err;
  }
  perm_scan_kernel<<<1, kScanThreads, 0, s>>>(hist, E, NW, counts, offsets, tile_offsets);
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

cudaError_t launch_scatter_rows_mx(const uint8_t* x_q, const uint8_t* x_scale, int T, int H,
                                   const int32_t* flat_to_perm, const int32_t* topk_idx,
                                   const int32_t* offsets, const int32_t* tile_offsets, int K, int TK,
                                   int E, uint8_t* x_perm, uint8_t* atoms, int* status,
                                   cudaStream_t s) {
  if (T == 0 || TK == 0) return cudaSuccess;
  if (H % 128) return cudaErrorInvalidValue;
  const int vecs = H / 16, nk = H / 128;
  const long long units = (long long)T * ((vecs + 127) / 128);
  const long long want = (units + 7) / 8;  // 8 warps a block
  const int blocks = want < 152 * 16 ? (int)want : 152 * 16;
  scatter_rows_mx_kernel<<<blocks, 256, 0, s>>>(
      reinterpret_cast<const uint4*>(x_q), reinterpret_cast<const uint32_t*>(x_scale), T, vecs, nk,
      flat_to_perm, topk_idx, offsets, tile_offsets, K, TK, E, reinterpret_cast<uint4*>(x_perm),
      reinterpret_cast<uint32_t*>(atoms), status);
  return cudaGetLastError();
}

}  // namespace moe
