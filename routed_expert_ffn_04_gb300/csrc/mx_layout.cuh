// Scale atoms: how E8M0 block scales (one per 32 elements along K) sit in
// memory for the block-scaled tensor cores.
//
// An atom holds the scales of a block of 128 rows x 128 K elements (4 per
// row) in 512 bytes: row r (0..127) of the block, K-block j (0..3) at byte
//   16 (r % 32) + 4 (r / 32) + j.
// Read as 32 rows of 16 bytes, that is the source tcgen05.cp 32x128b.warpx4
// copies into TMEM (replicated into all four lane quarters), where the
// tcgen05.mma kind::mxf8f6f4.block_scale (scale_vec::1X, M = N = 128) finds
// the scale of A row m in lane m, column m / 32, and that of B column n in
// column n / 32 of lane n % 32 of any quarter.
//
// A matrix of R rows (R % 128 == 0, or padded up to it) and K elements per row
// (K % 128 == 0) has (R / 128) x (K / 128) atoms, row-block major:
//   atom (R-block b, K-block a) at byte 512 (b (K / 128) + a).
#pragma once

#include <cstdint>

namespace moe {

constexpr int kAtomBytes = 512;

__host__ __device__ constexpr int atom_byte(int r, int j) {
  return 16 * (r & 31) + 4 * (r >> 5) + j;
}


}  // namespace moe
