// Step 3's GEMMs in MX formats with the weights on the MMA's M side: the same
// products as grouped_gemm_mx_kernel<MODE, W4> (gemm_mx.cu; "腾讯混元 Hy3 在
// CANN NPU 上的高性能推理部署与优化实战", section 8.2: W8A8 MXFP8 and the W4A8
// recipe with MXFP4 routed weights), tiled for few tokens per expert (decode).
//
// The token-tile kernels put 128 token rows of one expert on the M side of the
// MMA; at ~3 rows per expert nearly all of that tensor work is padding, and at
// N = 256 it is 536 cycles per K stage, most of the time a 16 KB E2M1 stage
// takes to stream from HBM. Here a tile is 256 weight rows (two M = 128 MMAs
// per K step) against up to 64 token rows of one expert as N = 64: per stage
// 8 MMAs of about 37 cycles of tensor work each, and only as many 16-row token
// boxes as the chunk has rows.
//   MODE 0 (GEMM-1): accumulator half s holds pair atom 2 wt + s of the
//                    gate/up rows (mx_layout.cuh order: TMEM lanes 0-63 gate,
//                    64-127 up, for 64 columns of h). SwiGLU pairs lane l
//                    with lane l + 64, which another warp reads, so the up
//                    lane quarters hand their values to the gate quarters
//                    through shared memory; the gate warps compute h and its
//                    MXFP8 codes: one E8M0 scale per 32 columns of a token,
//                    the 32 lanes of one warp.
//   MODE 1 (GEMM-2): 256 rows of W_down, y = h Wd^T for 256 columns, fp32,
//                    stored from registers (one 128-byte segment per token and
//                    warp).
//
// Scales travel in the atoms of the token-tile kernels (mx_layout.cuh): a
// chunk of 64 token rows is half of a 128-row activation atom, and the MMA
// finds the scale of B column n in column n / 32 of its scale address, so an
// odd chunk points the B scale address two columns into the atom.
//
// The pipeline is that of gemm_mx_wide.cu (one barrier wait per stage for an
// MMA thread, the weight ring, the token ring and the TMEM scale slot freed
// together by the MMA threads' commits; scale atoms two stages per bulk copy,
// two groups ahead), with two accumulators so that a tile's MMAs do not wait
// for the previous epilogue,
// and each CTA's first 64 tiles decoded once into shared memory, so that no
// role searches the group table at a tile boundary.
//
// Persistent, one CTA per SM, 416 threads:
//   warp 0      weight producer: per 128-wide K stage the tile's 256 weight
//               rows (one box for E2M1 in tile order, four for row-major
//               E4M3), 4-stage ring; the scale atoms of stage pairs; for
//               E2M1 GEMM-1 an L2 prefetch of the block four stages ahead.
//   warp 11     token producer: the chunk's rows in 16-row boxes, completing
//               on the weight stage's barrier.
//   warp 2      scale warp: three tcgen05.cp per stage into the stage's slot.
//   warps 1, 12 MMA issuers (warp 1 also allocates TMEM): 4 MMAs (K = 32)
//               each per stage, one per accumulator half.
//   warps 3-10  epilogue: warp w reads TMEM lane quarter w % 4 of accumulator
//               half (w - 3) / 4.
// TMEM: two accumulators of 2 x 64 columns, then one 16-column scale slot per
// stage (tokens +0..3, weight rows 0-127 +8..11, 128-255 +12..15).
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "gemm_sched.cuh"
#include "internal.h"
#include "mx.cuh"
#include "mx_layout.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int sStages = 4;                 // weight ring = token ring = TMEM scale slots
constexpr int sGroup = 2;                  // K stages per atom group (one bulk copy per atom kind)
constexpr int sGroupSlots = 4;             // atom groups in shared memory
constexpr int sGroupAhead = 2;             // groups between an atom group's load and its first stage
constexpr int sThreads = 416;
constexpr int sScaleWarp = 2;
constexpr int sEpiWarp0 = 3;
constexpr int sEpiWarps = 8;
constexpr int sProdTWarp = 11;
constexpr int sMmaWarp2 = 12;             // issues accumulator half 1's MMAs (warp 1 half 0's)
constexpr int sPrefetch = 4;               // E2M1 GEMM-1: L2 prefetch this many stages ahead of the ring
constexpr int sTokRows = 64;               // token rows per tile = MMA N
constexpr int sTokBox = 16;                // token rows per TMA box
constexpr int sTTile = sTokRows * 128;     // 64 token rows x 128 K bytes
constexpr int sWTile = 256 * 128;          // 256 weight rows x 128 K slots
constexpr int sBox = 64 * 128;             // one 64-row E4M3 weight box in shared memory
constexpr int sGroupBytes = 3 * sGroup * kAtomBytes;  // token atoms | weight atoms rows 0-127 | 128-255
constexpr int sAccCols = 2 * sTokRows;     // one accumulator: two halves of N columns
constexpr int sSfCol0 = 2 * sAccCols;      // TMEM scale slot s: sSfCol0 + 16 s
constexpr int sTmemCols = 512;
constexpr int sMaxGroups = 512;
constexpr int sTableStride = sMaxGroups + 8;
constexpr int sTileList = 64;              // a CTA's first tiles, decoded once in the prologue
constexpr int sTableBytes = 3 * sTableStride * 4 + sTileList * (int)sizeof(TileInfo);  // tile starts, row
                                           // starts, atom-block starts, the CTA's tile list
constexpr int sXchBlock = 32 * 32;         // fp32 values one up warp hands over per chunk
constexpr int sXchBytes = 4 * sXchBlock * 4;  // one block per gate/up quarter pair of each half
constexpr int sNumBars = 2 * sStages + 2 * sGroupSlots + 4 + 2 + 8 + 1;
constexpr int sBarBytes = 512;
// Shared memory: weight ring | token ring | atom groups | exchange | tables | barriers.
constexpr int sOffT = sStages * sWTile;
constexpr int sOffSf = sOffT + sStages * sTTile;
constexpr int sOffXch = sOffSf + sGroupSlots * sGroupBytes;
constexpr int sOffTable = sOffXch + sXchBytes;
constexpr int sOffBars = sOffTable + sTableBytes;
constexpr int sSmem = 1024 + sOffBars + sBarBytes;
static_assert(sSmem <= 232448, "shared memory budget");
static_assert(sSfCol0 + 16 * sStages <= sTmemCols, "TMEM budget");
static_assert(sNumBars * 8 + 8 <= sBarBytes, "barrier area");
static_assert(sTTile % 1024 == 0 && (sTokBox * 128) % 1024 == 0, "1024-byte alignment of swizzled token boxes");
static_assert(sOffXch % 16 == 0 && sOffTable % 16 == 0 && sOffBars % 8 == 0, "alignment");
static_assert(sTokRows % sTokBox == 0 && sTokRows == 64, "a chunk is half an activation atom");
static_assert(sThreads == 32 * (sMmaWarp2 + 1) && sProdTWarp + 1 == sMmaWarp2 && sEpiWarp0 + sEpiWarps == sProdTWarp,
              "warp roles");

// Parity of the phase of a ring barrier that completes for the n-th time
// (n = 0, 1, ...) when stage n * depth + slot completes.
__device__ __forceinline__ uint32_t round_parity(int stage, int depth) { return (uint32_t)(stage / depth) & 1u; }

// Prefetch `bytes` (a multiple of 16) from global address `src` (16-byte
// aligned) into L2, with no shared-memory destination.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Exclusive scan of v[0..n) in place by one warp; v[n] = the total.
__device__ __forceinline__ void warp_exclusive_scan(int32_t* v, int n, int lane) {
  const int per = (n + 31) / 32;
  const int b = lane * per;
  const int e = (b + per < n) ? b + per : n;
  int local = 0;
  for (int g = b; g < e; ++g) local += v[g];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  int run = incl - local;
  for (int g = b; g < e; ++g) {
    const int c = v[g];
    v[g] = run;
    run += c;
  }
  if (lane == 31) v[n] = incl;
}

// Bounded wait by every lane of a warp (each lane acquires the phase for its
// own reads); true when all lanes saw it complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t limit_ns) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, status, MOE_DEV_TIMEOUT_EPILOGUE, limit_ns);
  return __all_sync(0xFFFFFFFFu, ok) != 0;
}

// y for up to 32 tokens of one output column per lane: token j at y + j * ld.
__device__ __forceinline__ void store_y_tokens(const uint32_t (&v)[32], float* y, int n, int ld) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j < n) y[(size_t)j * ld] = __uint_as_float(v[j]);
}

// h for up to 32 tokens of 32 consecutive columns (one per lane): SwiGLU of
// the gate values g (this lane's column) and the up values u, then per token
// the MXFP8 block of the 32 lanes: shared exponent from the warp's amax, E4M3
// code per lane, E8M0 scale byte by lane 0. Token j is row row0 + j of h.
__device__ __forceinline__ void store_h_tokens(const uint32_t (&g)[32], const float (&u)[32], int n,
                                               uint8_t* h_col, int ld, int r_first, int lane,
                                               uint8_t* scale_blk0, int blocks_per_atom_row, int jcol) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < n) {
      const float hv = silu_f(__uint_as_float(g[j])) * u[j];
      float amax = fabsf(hv);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      uint32_t code = 0, sc = 0;
      if (amax != 0.0f) {
        const int sexp = mx_shared_exp(amax);
        code = mx_encode(hv, sexp);
        sc = (uint32_t)(sexp + 127);
      }
      h_col[(size_t)j * ld] = (uint8_t)code;
      if (lane == 0) {
        const int r = r_first + j;  // row of the token within its group
        scale_blk0[(size_t)(r >> 7) * blocks_per_atom_row * kAtomBytes + atom_byte(r & 127, jcol)] = (uint8_t)sc;
      }
    }
  }
}

template <int MODE, bool W4>
__global__ void __launch_bounds__(sThreads, 1)
    grouped_gemm_mx_swap_kernel(const __grid_constant__ CUtensorMap map_act,
                                const __grid_constant__ CUtensorMap map_w0,
                                const __grid_constant__ CUtensorMap map_w1, const KParams p,
                                const uint8_t* __restrict__ w_tiled) {
  // Weight transaction bytes of a stage (E2M1 boxes count their packed global
  // bytes, half their shared-memory footprint); the token boxes add 2 KB each.
  constexpr uint32_t kTxW = W4 ? sWTile / 2 : sWTile;
  constexpr uint32_t kTxBox = sTokBox * 128;
  // A = weights (format E2M1 or E4M3), B = tokens (E4M3), M = 128, N = 64.
  constexpr uint32_t kIdesc0 = idesc_mxf8_e4m3(128, sTokRows, 0, 0) | (W4 ? (5u << 7) : 0u);
  // Output columns per tile: GEMM-1 128 of h (256 gate/up rows), GEMM-2 256 of y.
  constexpr int kCols = MODE == 0 ? 128 : 256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* base = smem_raw + pad;
  const uint32_t sm0 = raw_addr + pad;
  float* xch = reinterpret_cast<float*>(base + sOffXch);
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + sOffTable);
  int32_t* row_start = tile_start + sTableStride;
  int32_t* blk_start = row_start + sTableStride;
  TileInfo* tlist = reinterpret_cast<TileInfo*>(blk_start + sTableStride);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + sOffBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + sNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // full(s): stage s's weights and tokens landed and its scales are in TMEM
  // slot s (two arrivals: the weight producer's, with both producers' bytes,
  // and the scale warp's commit); empty(s): its MMAs are done (frees the
  // weight stage, the token stage and TMEM scale slot s).
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (sStages + s); };
  // gfull(g): atom group slot g landed; gfree(g): its copies into TMEM are done.
  auto gfull = [&](int g) { return bar0 + 8u * (2 * sStages + g); };
  auto gfree = [&](int g) { return bar0 + 8u * (2 * sStages + sGroupSlots + g); };
  const uint32_t tbar0 = bar0 + 8u * (2 * sStages + 2 * sGroupSlots);
  auto tfull = [&](int a) { return tbar0 + 8u * a; };
  auto tempty = [&](int a) { return tbar0 + 8u * (2 + a); };
  const uint32_t drain_bar = tbar0 + 32u;
  const uint32_t sdrain_bar = tbar0 + 40u;
  // GEMM-1 exchange slot x (half x / 2, gate/up quarter pair x % 2): xfull
  // when the up warp wrote a chunk, xfree when the gate warp read it.
  auto xfull = [&](int x) { return tbar0 + 48u + 8u * x; };
  auto xfree = [&](int x) { return tbar0 + 80u + 8u * x; };
  const uint32_t drain_bar2 = tbar0 + 112u;  // the second MMA thread's drain

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_wt = p.N / kCols;
  fill_row_start(p, row_start, threadIdx.x, sThreads);
  for (int g = threadIdx.x; g < p.G; g += sThreads) {
    int r0, nr;
    group_rows(p, g, r0, nr);
    tile_start[g] = n_wt * ((nr + sTokRows - 1) / sTokRows);
    blk_start[g] = (nr + 127) / 128;  // the group's 128-row activation atom blocks
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < sStages; ++s) {
      mbar_init(full(s), 2);
      mbar_init(empty(s), 2);  // one commit from each MMA thread
    }
    for (int g = 0; g < sGroupSlots; ++g) {
      mbar_init(gfull(g), 1);
      mbar_init(gfree(g), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 2);
      mbar_init(tempty(a), sEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(drain_bar2, 1);
    mbar_init(sdrain_bar, 1);
    for (int x = 0; x < 4; ++x) {
      mbar_init(xfull(x), 32);
      mbar_init(xfree(x), 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), sTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_act);
    prefetch_tensormap(&map_w0);
    prefetch_tensormap(&map_w1);
  }
  __syncthreads();
  if (warp == 0) warp_exclusive_scan(tile_start, p.G, lane);
  if (warp == 2) warp_exclusive_scan(blk_start, p.G, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[p.G];
  const int n_k = p.num_kb / 2;  // p.num_kb counts 64-wide slices; a stage holds two
  // The CTA's k-th tile (blockIdx.x + k * gridDim.x), decoded once here for the
  // first sTileList: a role starting a tile then reads it from shared memory
  // instead of searching the group table (a tile boundary cost the MMA thread
  // about a stage's time, the weight producer three).
  for (int k = threadIdx.x; k < sTileList; k += sThreads) {
    const int tile = blockIdx.x + k * (int)gridDim.x;
    if (tile < total) tlist[k] = decode_tile_s<sTokRows>(p.G, tile_start, row_start, tile);
  }
  __syncthreads();
  auto tile_info = [&](int k, int tile) -> TileInfo {
    return k < sTileList ? tlist[k] : decode_tile_s<sTokRows>(p.G, tile_start, row_start, tile);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();   // each weight byte is read once
      const uint64_t pol_t = l2_policy_evict_normal();  // token atoms: every weight tile of the expert
      Armed armed, armed_g;
      bool ok = true;
      // Atom groups: a group is up to sGroup consecutive K stages of one tile.
      int g_tile = blockIdx.x, g_k = 0, g_kb = 0, nload = 0;
      TileInfo g_ti{};
      if (g_tile < total) g_ti = tile_info(0, g_tile);
      auto load_group = [&]() -> bool {
        if (g_tile >= total) return true;
        const int gs = nload % sGroupSlots;
        if (nload >= sGroupSlots &&
            !mbar_wait_bounded(gfree(gs), round_parity(nload - sGroupSlots, sGroupSlots), abort_flag, p.status,
                               MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns))
          return false;
        const int cnt = n_k - g_kb < sGroup ? n_k - g_kb : sGroup;
        const uint32_t bytes = (uint32_t)cnt * kAtomBytes;
        // Token atoms: the activation atom block holding the chunk. Weight
        // atoms b_blk, b_blk + 1: GEMM-1 the gate/up atom matrix (2N rows per
        // group), GEMM-2 the down atoms (N rows per group).
        const long long a_blk = blk_start[g_ti.g] + g_ti.tt / 2;
        const long long b_blk = (long long)g_ti.g * ((MODE == 0 ? 2 : 1) * p.N / 128) + 2 * g_ti.wt;
        const uint8_t* a_atom = p.s_act + (a_blk * n_k + g_kb) * kAtomBytes;
        const uint8_t* b_atom = p.s_w0 + (b_blk * n_k + g_kb) * kAtomBytes;
        const uint32_t dst = sm0 + sOffSf + gs * sGroupBytes;
        const uint32_t fb = gfull(gs);
        mbar_arrive_expect_tx(fb, 3 * bytes);
        bulk_load_hint(dst, a_atom, bytes, fb, pol_t);
        bulk_load_hint(dst + sGroup * kAtomBytes, b_atom, bytes, fb, pol_w);
        bulk_load_hint(dst + 2 * sGroup * kAtomBytes, b_atom + (size_t)n_k * kAtomBytes, bytes, fb, pol_w);
        Ring at;
        at.s = gs;
        at.ph = round_parity(nload, sGroupSlots);
        armed_g.mark(at);
        ++nload;
        g_kb += cnt;
        if (g_kb == n_k) {
          g_kb = 0;
          g_tile += gridDim.x;
          ++g_k;
          if (g_tile < total) g_ti = tile_info(g_k, g_tile);
        }
        return true;
      };
      // GEMM-1 with E2M1 weights in tile order: the ring holds 16 KB of weights
      // per stage, few bytes in flight per SM, so the block of the stage
      // sPrefetch ahead (tile-order block t of K block kb: 256 rows of 64
      // bytes) is also requested into L2: decode shape 0.210 -> 0.204 ms. For
      // GEMM-2 (two 128-row blocks a stage) the two extra requests measured
      // slower (0.118 -> 0.128 ms), so it has none.
      constexpr int kPrefetch = MODE == 0 ? sPrefetch : 0;
      auto prefetch_stage = [&](int t_, int kb_) {
        constexpr uint32_t kBlk = 256 * 64;
        bulk_prefetch_l2(w_tiled + ((size_t)t_ * n_k + kb_) * kBlk, kBlk);
      };
      auto block_of = [&](const TileInfo& ti) {
        return MODE == 0 ? ti.g * n_wt + ti.wt : (ti.g * p.N + ti.wt * kCols) / 128;
      };
      for (int i = 0; ok && i < sGroupAhead; ++i) ok = load_group();
      int j = 0;  // stage
      for (int tile = blockIdx.x, k = 0; ok && tile < total; tile += gridDim.x, ++k) {
        const TileInfo ti = tile_info(k, tile);
        const int w_row = ti.g * p.N + ti.wt * kCols;
        // Tile order: GEMM-1 the gate/up pair block t (256 rows), GEMM-2 the
        // 128-row down blocks t and t + 1.
        const int t = block_of(ti);
        const bool has_next = tile + (int)gridDim.x < total;
        const int t_next =
            has_next ? block_of(tile_info(k + 1, tile + gridDim.x)) : 0;
        const int rem = ti.nrows - ti.tt * sTokRows;
        const int nb = ((rem < sTokRows ? rem : sTokRows) + sTokBox - 1) / sTokBox;
        const uint32_t tx = kTxW + (uint32_t)nb * kTxBox;
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          if (kb % sGroup == 0 && !load_group()) {
            ok = false;
            break;
          }
          const int s = j % sStages;
          if (j >= sStages && !mbar_wait_bounded(empty(s), round_parity(j - sStages, sStages), abort_flag,
                                                 p.status, MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full(s);
          mbar_arrive_expect_tx(fb, tx);
          const uint32_t st = sm0 + s * sWTile;
          if (W4) {
            if (MODE == 0) {
              tma_load_2d_hint(st, &map_w0, fb, 0, (t * n_k + kb) * 256, pol_w);
            } else {
              tma_load_2d_hint(st, &map_w0, fb, 0, (t * n_k + kb) * 128, pol_w);
              tma_load_2d_hint(st + 2 * sBox, &map_w0, fb, 0, ((t + 1) * n_k + kb) * 128, pol_w);
            }
            if (kPrefetch > 0) {
              const int kp = kb + kPrefetch;
              if (kp < n_k) prefetch_stage(t, kp);
              else if (has_next && kp - n_k < n_k) prefetch_stage(t_next, kp - n_k);
            }
          } else {
            // Row-major E4M3, four 64-row boxes: GEMM-1 gate, up, gate, up (64 rows
            // each, the atoms' order); GEMM-2 256 consecutive down rows.
            const int kx = kb * 128;
            const CUtensorMap* m1 = MODE == 0 ? &map_w1 : &map_w0;
            const int r1 = MODE == 0 ? 0 : 64;
            tma_load_2d_hint(st, &map_w0, fb, kx, w_row, pol_w);
            tma_load_2d_hint(st + sBox, m1, fb, kx, w_row + r1, pol_w);
            tma_load_2d_hint(st + 2 * sBox, &map_w0, fb, kx, w_row + (MODE == 0 ? 64 : 128), pol_w);
            tma_load_2d_hint(st + 3 * sBox, m1, fb, kx, w_row + (MODE == 0 ? 64 : 192), pol_w);
          }
          Ring r;
          r.s = s;
          r.ph = round_parity(j, sStages);
          armed.mark(r);
        }
      }
      if (!ok) {
        for (int s = 0; s < sStages; ++s)
          if (armed.mask & (1u << s)) drain_wait(full(s), (armed.phase >> s) & 1u, 100000000ull);
        for (int g = 0; g < sGroupSlots; ++g)
          if (armed_g.mask & (1u << g)) drain_wait(gfull(g), (armed_g.phase >> g) & 1u, 100000000ull);
      }
    }
  } else if (warp == sProdTWarp) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      bool ok = true;
      Armed armed;
      int j = 0;
      for (int tile = blockIdx.x, k = 0; ok && tile < total; tile += gridDim.x, ++k) {
        const TileInfo ti = tile_info(k, tile);
        const int row = ti.row0 + ti.tt * sTokRows;
        const int rem = ti.nrows - ti.tt * sTokRows;
        const int nb = ((rem < sTokRows ? rem : sTokRows) + sTokBox - 1) / sTokBox;
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          // Token slot j % sStages last held stage j - sStages, whose MMAs
          // completed empty(j % sStages); the phase of full(j % sStages) these
          // loads complete on is then the current one.
          if (j >= sStages && !mbar_wait_bounded(empty(j % sStages), round_parity(j - sStages, sStages),
                                                 abort_flag, p.status, MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t dst = sm0 + sOffT + (j % sStages) * sTTile;
          for (int b = 0; b < nb; ++b)
            tma_load_2d(dst + b * kTxBox, &map_act, full(j % sStages), kb * 128, row + b * sTokBox);
          Ring r;
          r.s = j % sStages;
          r.ph = round_parity(j, sStages);
          armed.mark(r);
        }
      }
      if (!ok) {  // bounded: a stage the weight producer never armed does not complete
        for (int s = 0; s < sStages; ++s)
          if (armed.mask & (1u << s)) drain_wait(full(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == sScaleWarp) {
    // ------------------------------------------------------------ scale warp
    if (lane == 0) {
      bool ok = true, issued = false;
      int j = 0, ng = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          const int gs = ng % sGroupSlots;
          const int i = kb % sGroup;  // stage within its atom group
          const bool last = i == sGroup - 1 || kb == n_k - 1;
          const int s = j % sStages;
          // The group's atoms have landed; TMEM slot s is free once the MMAs
          // of stage j - sStages are done.
          if ((i == 0 && !mbar_wait_bounded(gfull(gs), round_parity(ng, sGroupSlots), abort_flag, p.status,
                                            MOE_DEV_TIMEOUT_MMA, p.limit_ns)) ||
              (j >= sStages && !mbar_wait_bounded(empty(s), round_parity(j - sStages, sStages), abort_flag,
                                                  p.status, MOE_DEV_TIMEOUT_MMA, p.limit_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tmem_base + (uint32_t)(sSfCol0 + 16 * s);
          const uint32_t src = sm0 + sOffSf + gs * sGroupBytes + i * kAtomBytes;
          tmem_cp_32x128b_warpx4(sf, src);
          tmem_cp_32x128b_warpx4(sf + 8, src + sGroup * kAtomBytes);
          tmem_cp_32x128b_warpx4(sf + 12, src + 2 * sGroup * kAtomBytes);
          issued = true;
          umma_commit(full(s));
          if (last) {
            umma_commit(gfree(gs));  // the group slot may be reloaded once these copies are done
            ++ng;
          }
        }
      }
      if (!ok && issued) {  // its copies complete before TMEM is freed
        umma_commit(sdrain_bar);
        drain_wait(sdrain_bar, 0, 100000000ull);
      }
    }
  } else if (warp == 1 || warp == sMmaWarp2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues accumulator half 0's MMAs, warp sMmaWarp2 half 1's: each
    // tcgen05.mma costs its issuing thread ~55 cycles, 8 a stage were most of
    // one thread's stage time. Each commits to empty(s) and tfull (count 2).
    if (lane == 0) {
      const int hsel = warp == 1 ? 0 : 1;
      const uint32_t drain = hsel ? drain_bar2 : drain_bar;
      bool ok = true, issued = false;
      int local = 0, j = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t ap = (uint32_t)(local >> 1) & 1u;
        if (!mbar_wait_bounded(tempty(acc), ap ^ 1u, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA, p.limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const TileInfo ti = tile_info(local, tile);
        const uint32_t d = tmem_base + (uint32_t)(acc * sAccCols + hsel * sTokRows);
        const uint32_t sfb_col = 2u * (uint32_t)(ti.tt & 1);  // odd chunks: rows 64-127 of the token atom
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          const int s = j % sStages;
          if (!mbar_wait_bounded(full(s), round_parity(j, sStages), abort_flag, p.status, MOE_DEV_TIMEOUT_MMA,
                                 p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // +32 bytes along K is +2 in a descriptor's start-address field.
          const uint64_t dt = sw128_kmajor_desc(sm0 + sOffT + s * sTTile);
          const uint64_t dw = sw128_kmajor_desc(sm0 + s * sWTile + hsel * (128 * 128));  // weight rows 128 hsel..
          const uint32_t sf = tmem_base + (uint32_t)(sSfCol0 + 16 * s);
          const uint32_t sfa = sf + 8 + 4 * hsel;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // Scale ids (bits 4-5 for B, 29-30 for A) pick byte k of the scale words.
            const uint32_t id = kIdesc0 | ((uint32_t)k << 4) | ((uint32_t)k << 29);
            umma_mxf8(d, dw + 2 * k, dt + 2 * k, id, sfa, sf + sfb_col, (kb | k) ? 1u : 0u);
          }
          issued = true;
          umma_commit(empty(s));
        }
        if (!ok) break;
        umma_commit(tfull(acc));
      }
      if (!ok && issued) {
        umma_commit(drain);
        drain_wait(drain, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quarter this warp may read
    const int hf = (warp - sEpiWarp0) >> 2;    // accumulator half
    const int xi = hf * 2 + (q & 1);           // GEMM-1 exchange slot of this gate/up quarter pair
    float* xb = xch + xi * sXchBlock;
    int local = 0, e = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t ap = (uint32_t)(local >> 1) & 1u;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull(acc), ap, abort_flag, p.status, MOE_DEV_TIMEOUT_EPILOGUE, p.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = tile_info(local, tile);
      const int r_first = ti.tt * sTokRows;  // first token row of the chunk within its group
      const int rem = ti.nrows - r_first;
      const int ncols = rem < sTokRows ? rem : sTokRows;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * sAccCols + hf * sTokRows);
      uint32_t v0[32], v1[32];
      tmem_ld_32x32b_x32(tb, v0);
      if (ncols > 32) tmem_ld_32x32b_x32(tb + 32, v1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));  // the MMA may overwrite this accumulator now
      if (MODE == 1) {
        float* y = static_cast<float*>(p.out) + (size_t)(ti.row0 + r_first) * p.N + ti.wt * kCols +
                   hf * 128 + q * 32 + lane;
        store_y_tokens(v0, y, ncols, p.N);
        if (ncols > 32) store_y_tokens(v1, y + (size_t)32 * p.N, ncols - 32, p.N);
      } else {
        // Lanes 64-127 of a half (quarters 2, 3) hold the up rows of the gate
        // rows in lanes 0-63 (quarters 0, 1): one 32 x 32 block per chunk goes
        // from the up warp to the gate warp of its pair.
        const int col = ti.wt * 128 + hf * 64 + 32 * (q & 1);  // first h column of this pair
        uint8_t* h_col = static_cast<uint8_t*>(p.out) + (size_t)(ti.row0 + r_first) * p.N + col + lane;
        uint8_t* scale_blk0 = p.out_scale + ((size_t)blk_start[ti.g] * (p.N / 128) + ti.wt) * kAtomBytes;
        const int jcol = (col / 32) & 3;
        auto chunk = [&](const uint32_t (&v)[32], int c) -> bool {
          const int n = ncols - 32 * c;
          if (q >= 2) {
            if (e > 0 && !warp_wait(xfree(xi), (uint32_t)(e - 1) & 1u, abort_flag, p.status, p.limit_ns))
              return false;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (jj < n) xb[jj * 32 + lane] = __uint_as_float(v[jj]);
            mbar_arrive(xfull(xi));
          } else {
            if (!warp_wait(xfull(xi), (uint32_t)e & 1u, abort_flag, p.status, p.limit_ns)) return false;
            float u[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) u[jj] = jj < n ? xb[jj * 32 + lane] : 0.0f;
            mbar_arrive(xfree(xi));
            store_h_tokens(v, u, n, h_col + (size_t)(32 * c) * p.N, p.N, r_first + 32 * c, lane, scale_blk0,
                           p.N / 128, jcol);
          }
          ++e;
          return true;
        };
        if (!chunk(v0, 0)) break;
        if (ncols > 32 && !chunk(v1, 1)) break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, sTmemCols);
  }
}

template <int MODE, bool W4>
cudaError_t run_gemm_mx_swap(const GroupedGemmArgs& a, cudaStream_t s) {
  if (a.rows == 0 || a.G == 0) return cudaSuccess;
  if (a.H % 128 || a.I % 128 || a.G > sMaxGroups || (MODE == 1 && a.H % 256)) return cudaErrorInvalidValue;
  const int G = a.offsets ? a.G : 1;
  const int Kdim = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const void* act = MODE == 0 ? a.a : a.h;
  CUtensorMap m_act, m_w0, m_w1;
  bool maps_ok = make_tmap_u8(&m_act, act, Kdim, a.rows, sTokBox);
  if (W4) {  // tile order: GEMM-1 the gate/up pair (256-row boxes), GEMM-2 down (128-row boxes)
    maps_ok = maps_ok && (MODE == 0 ? make_tmap_e2m1(&m_w0, a.w_gate, 2ull * G * N * (Kdim / 128), 256)
                                    : make_tmap_e2m1(&m_w0, a.w_down, (uint64_t)G * N * (Kdim / 128), 128));
    m_w1 = m_w0;
  } else if (MODE == 0) {
    maps_ok = maps_ok && make_tmap_u8(&m_w0, a.w_gate, Kdim, (uint64_t)G * N, 64) &&
              make_tmap_u8(&m_w1, a.w_up, Kdim, (uint64_t)G * N, 64);
  } else {
    maps_ok = maps_ok && make_tmap_u8(&m_w0, a.w_down, Kdim, (uint64_t)G * N, 64);
    m_w1 = m_w0;
  }
  if (!maps_ok) return cudaErrorInvalidValue;
  KParams p = {};
  p.offsets = a.offsets;
  p.G = G;
  p.rows = a.rows;
  p.num_kb = Kdim / 64;
  p.N = N;
  p.out = MODE == 0 ? a.h : static_cast<void*>(a.y);
  p.status = a.status;
  p.limit_ns = a.wait_limit_ns;
  p.s_w0 = MODE == 0 ? a.s_gate : a.s_down;
  p.s_act = MODE == 0 ? a.a_scale : a.h_scale;
  p.out_scale = MODE == 0 ? a.h_scale : nullptr;
  const long long n_wt = N / (MODE == 0 ? 128 : 256);
  const long long max_tiles = n_wt * ((a.rows + sTokRows - 1) / sTokRows + G);
  const int grid = (int)(max_tiles < a.num_sms ? max_tiles : a.num_sms);
  const uint8_t* w_tiled = static_cast<const uint8_t*>(MODE == 0 ? a.w_gate : a.w_down);
  grouped_gemm_mx_swap_kernel<MODE, W4><<<grid, sThreads, sSmem, s>>>(m_act, m_w0, m_w1, p, w_tiled);
  return cudaGetLastError();
}

}  // namespace

bool gemm_mx_swap_supported(const GroupedGemmArgs& a, int mode) {
  return (a.offsets ? a.G : 1) <= sMaxGroups && (mode == 0 || a.H % 256 == 0);
}

cudaError_t gemm_mx_swap_prepare_device() {
  const cudaError_t errs[] = {
      cudaFuncSetAttribute(grouped_gemm_mx_swap_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_swap_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_swap_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, sSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_swap_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, sSmem)};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_gemm_mx_swap_gate_up(const GroupedGemmArgs& a, cudaStream_t s) {
  return a.w4 ? run_gemm_mx_swap<0, true>(a, s) : run_gemm_mx_swap<0, false>(a, s);
}

cudaError_t launch_gemm_mx_swap_down(const GroupedGemmArgs& a, cudaStream_t s) {
  return a.w4 ? run_gemm_mx_swap<1, true>(a, s) : run_gemm_mx_swap<1, false>(a, s);
}

}  // namespace moe
