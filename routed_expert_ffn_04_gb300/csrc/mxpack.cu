// Scale atoms (mx_layout.cuh) for the block-scaled MXFP8 GEMM: packing of
// row-major E8M0 weight scales, and the gather of activation scales into one
// atom row-block per token tile of each expert group. Also the tile order of
// packed E2M1 weights (the W4A8 routed experts).
//
// Weights ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section
// 8.2: routed and shared expert Linears in MXFP8) are packed once, like their
// quantisation. Gate and up are packed together: the atom matrix interleaves
// them per 64 rows (gate rows 0..63, up rows 0..63, gate rows 64..127, ...),
// which is the row order of one GEMM-1 tile (64 gate + 64 up outputs).
#include <cuda_runtime.h>

#include "internal.h"
#include "mx_layout.cuh"

namespace moe {
namespace {

// One thread per 4-byte atom word (the word of atom a at byte 4 (w & 127)
// holds the 4 scales of block row 32 (j % 4) + j / 4, j = w % 128).
__global__ void __launch_bounds__(256) pack_weight_scales_kernel(const uint8_t* __restrict__ s0,
                                                                 const uint8_t* __restrict__ s1,
                                                                 long long words, int nk,
                                                                 int row_bytes,
                                                                 uint32_t* __restrict__ out) {
  const long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= words) return;
  const long long a = w >> 7;
  const int j = (int)(w & 127);
  const long long v = (a / nk) * 128 + 32 * (j & 3) + (j >> 2);  // row of the atom matrix
  const int ka = (int)(a % nk);
  const uint8_t* src = s0;
  long long row = v;
  if (s1) {  // gate/up interleave per 64 rows
    src = ((v >> 6) & 1) ? s1 : s0;
    row = (v >> 7) * 64 + (v & 63);
  }
  out[w] = __ldg(reinterpret_cast<const uint32_t*>(src + row * row_bytes) + ka);
}

constexpr int kGatherThreads = 256;
constexpr int kMaxGroups = 1024;

// out: atoms of the activation scales, one atom row-block per 128 rows of a
// group (the group's token tiles, in group order). Row j of group g is
// src row perm_src[row0_g + j] / K (or row0_g + j without perm_src). Rows of
// a group's last tile past its end are left untouched.
__global__ void __launch_bounds__(kGatherThreads) gather_scale_atoms_kernel(
    const uint8_t* __restrict__ src, int src_rows, int row_bytes, int nk,
    const int32_t* __restrict__ perm_src, int K, const int32_t* __restrict__ offsets, int G,
    int rows, uint32_t* __restrict__ out, int* status) {
  __shared__ int row0[kMaxGroups];
  __shared__ int item0[kMaxGroups + 1];  // first row item of each group
  __shared__ int tile0[kMaxGroups];      // first token tile of each group
  __shared__ int part_items[kGatherThreads], part_tiles[kGatherThreads];
  const int tid = threadIdx.x;
  // Clamped group bounds, as the grouped GEMM reads them.
  const int per = (G + kGatherThreads - 1) / kGatherThreads;
  const int gb = tid * per, ge = gb + per < G ? gb + per : G;
  int si = 0, st = 0;
  for (int g = gb; g < ge; ++g) {
    int a = 0, b = rows;
    if (offsets) {
      a = __ldg(offsets + g);
      b = __ldg(offsets + g + 1);
      a = a < 0 ? 0 : (a > rows ? rows : a);
      b = b < a ? a : (b > rows ? rows : b);
    }
    row0[g] = a;
    item0[g] = b - a;  // count for now
    si += b - a;
    st += (b - a + 127) / 128;
  }
  part_items[tid] = si;
  part_tiles[tid] = st;
  __syncthreads();
  if (tid == 0) {
    int ri = 0, rt = 0;
    for (int t = 0; t < kGatherThreads; ++t) {
      const int ci = part_items[t], ct = part_tiles[t];
      part_items[t] = ri;
      part_tiles[t] = rt;
      ri += ci;
      rt += ct;
    }
    item0[G] = ri;
  }
  __syncthreads();
  {
    int ri = part_items[tid], rt = part_tiles[tid];
    for (int g = gb; g < ge; ++g) {
      const int c = item0[g];
      item0[g] = ri;
      tile0[g] = rt;
      ri += c;
      rt += (c + 127) / 128;
    }
  }
  __syncthreads();
  const long long total = (long long)item0[G] * nk;
  for (long long it = (long long)blockIdx.x * blockDim.x + tid; it < total;
       it += (long long)gridDim.x * blockDim.x) {
    const int u = (int)(it / nk), ka = (int)(it % nk);
    int lo = 0, hi = G;  // item0[lo] <= u < item0[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (item0[mid] <= u) lo = mid; else hi = mid;
    }
    const int j = u - item0[lo];
    const int r = row0[lo] + j;
    int t = r;
    if (perm_src) {
      const int f = __ldg(perm_src + r);
      t = ((unsigned)f < (unsigned)rows) ? f / K : -1;
    }
    uint32_t v = 0u;  // finite scale (2^-127) for a row that has no source
    if (t >= 0 && t < src_rows)
      v = __ldg(reinterpret_cast<const uint32_t*>(src + (size_t)t * row_bytes) + ka);
    else if (ka == 0)
      atomicCAS(status, 0, MOE_DEV_BAD_PERM_INDEX);
    const long long blk = tile0[lo] + j / 128;
    out[((blk * nk + ka) * kAtomBytes + atom_byte(j & 127, 0)) / 4] = v;
  }
}

// Packed E2M1 weights [rows, cols/2] -> tile order (moe_tile_mxfp4_weights):
// per 128-row block t and 128-element K block kb one contiguous block at
// (t * nk + kb): 128 rows of 64 bytes (q1 == nullptr, 8 KB), or for a gate
// (q0) / up (q1) pair 16 KB: q0 rows 0-63, q1 rows 0-63, q0 rows 64-127, q1
// rows 64-127 of the block. One thread per 16 bytes of the output.
__global__ void __launch_bounds__(256) tile_e2m1_kernel(const uint4* __restrict__ q0, const uint4* __restrict__ q1,
                                                        long long chunks, int nk, uint4* __restrict__ dst) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= chunks) return;
  const int per_blk = q1 ? 1024 : 512;  // 16-byte chunks per block
  const long long blk = i / per_blk;
  const int within = (int)(i - blk * per_blk);
  const long long t = blk / nk;
  const int kb = (int)(blk - t * nk);
  const uint4* src = q0;
  int r = within >> 2;
  if (q1) {
    const int quarter = within >> 8;  // 64-row pieces: q0, q1, q0, q1
    src = (quarter & 1) ? q1 : q0;
    r = (quarter >> 1) * 64 + ((within & 255) >> 2);
  }
  // Source row: nk * 4 chunks of 16 bytes; this block's 64 bytes start at chunk 4 kb.
  dst[i] = __ldg(src + (t * 128 + r) * (nk * 4) + kb * 4 + (within & 3));
}

}  // namespace

cudaError_t launch_tile_e2m1(const uint8_t* q0, const uint8_t* q1, int64_t rows, int cols, uint8_t* dst,
                             cudaStream_t s) {
  const long long chunks = (q1 ? 2 : 1) * (long long)rows * cols / 32;  // bytes / 16
  if (chunks == 0) return cudaSuccess;
  tile_e2m1_kernel<<<(unsigned)((chunks + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(q0), reinterpret_cast<const uint4*>(q1), chunks, cols / 128,
      reinterpret_cast<uint4*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_pack_weight_scales(const uint8_t* s0, const uint8_t* s1, int64_t rows, int cols,
                                      uint8_t* out, cudaStream_t s) {
  const int nk = cols / 128;
  const long long vrows = s1 ? 2 * rows : rows;
  const long long words = vrows / 128 * nk * 128;
  if (words == 0) return cudaSuccess;
  const long long grid = (words + 255) / 256;
  pack_weight_scales_kernel<<<(unsigned)grid, 256, 0, s>>>(s0, s1, words, nk, cols / 32,
                                                           reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_gather_scale_atoms(const uint8_t* src, int src_rows, int cols,
                                      const int32_t* perm_src, int K, const int32_t* offsets,
                                      int G, int rows, uint8_t* out, int* status, cudaStream_t s) {
  if (rows == 0 || G == 0) return cudaSuccess;
  if (G > kMaxGroups || cols % 128) return cudaErrorInvalidValue;
  const int nk = cols / 128;
  long long blocks = ((long long)rows * nk + kGatherThreads - 1) / kGatherThreads;
  if (blocks > 152 * 4) blocks = 152 * 4;
  gather_scale_atoms_kernel<<<(unsigned)blocks, kGatherThreads, 0, s>>>(
      src, src_rows, cols / 32, nk, perm_src, K, offsets, offsets ? G : 1, rows,
      reinterpret_cast<uint32_t*>(out), status);
  return cudaGetLastError();
}

size_t scale_atom_bytes(int64_t rows, int groups, int cols) {
  return (size_t)(rows / 128 + groups) * (cols / 128) * kAtomBytes;
}

}  // namespace moe
