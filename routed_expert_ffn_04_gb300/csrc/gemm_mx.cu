// Step 3 in MXFP8 on the block-scaled tensor cores: the grouped SwiGLU
// expert GEMM with E4M3 activations and weights and one E8M0 scale per 32
// elements along K ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战",
// section 8.2: routed and shared Linears in W8A8 MXFP8). The MMA is
// tcgen05.mma kind::mxf8f6f4.block_scale: the tensor cores apply the scales,
// so nothing is expanded to bf16 on the way.
//
//   GEMM-1 (MODE 0): h = silu(x Wg^T) * (x Wu^T), re-quantised to MXFP8 per
//                    32 along I and stored as E4M3 codes + E8M0 scales
//   GEMM-2 (MODE 1): y = h Wd^T, fp32
//
// W4 (the W4A8 recipe of the same section: MXFP4 routed-expert weights, MXFP8
// activations): the weights are packed E2M1 in tile order
// (moe_tile_mxfp4_weights: a stage's 128 weight rows are one contiguous block,
// one TMA load), loaded through a 16U4 tensor map that puts each 16 codes in
// the low half of a 16-byte slot, the operand layout kind::mxf8f6f4 reads for
// E2M1 (B format code 5). Shared-memory tiles, scales and the MMA shape are
// those of E4M3; HBM weight bytes halve.
//
// Scales travel in scale atoms (mx_layout.cuh): 512 bytes per 128 rows x 128
// K elements, already in the order the block-scaled MMA reads from TMEM.
// A stage's two atoms (A rows, B rows) ride on the same mbarrier as its TMA
// tiles, and the MMA thread moves them into TMEM with tcgen05.cp.
//
// Persistent, one CTA per SM, 224 threads:
//   warp 0      producer: per stage, the 128-wide K slice (bytes) of the 128
//               token rows (A) and 128 weight rows (B) by TMA, plus the two
//               scale atoms by bulk copy.
//   warp 6      scale mover: per stage, once the stage has landed, two
//               tcgen05.cp (32x128b.warpx4: one 32 x 16-byte atom block
//               replicated into the four lane quarters) into the stage's TMEM
//               scale slot, committed to the stage's scale barrier.
//   warp 1      TMEM allocator + MMA issuer: per stage, after the scale
//               barrier, 4 MMAs (K = 32 each). Each tcgen05 instruction costs
//               its issuing thread tens of cycles, and at N = 128 the MMA
//               thread's issue time, not the tensor pipe, sets the pace, so
//               the copies are issued by another thread.
//   warps 2..5  epilogue (TMEM -> h codes + scale atoms, or staged fp32 y).
// Tile: M = 128 tokens, N = 128 (GEMM-1: gate 64 + up 64; GEMM-2: 128 of
// H), double-buffered fp32 accumulators (256 TMEM columns) plus one 8-column
// scale slot per stage.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "gemm_sched.cuh"
#include "internal.h"
#include "mx.cuh"
#include "mx_layout.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kK = 128;                  // K elements (= bytes) per stage
constexpr int kStages = 6;
constexpr int kThreads = 224;
constexpr int kMoverWarp = 6;
constexpr int kTileBytes = 128 * 128;    // 128 rows x 128 bytes
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kSfBytes = 2 * kAtomBytes; // per stage: A atom + B atom
constexpr int kAccCols = 128;
constexpr int kSfCol0 = 2 * kAccCols;    // scale slot of stage s: kSfCol0 + 8 s (A: +0..3, B: +4..7)
constexpr int kTmemCols = 512;
constexpr int kMaxGroups = 1024;
constexpr int kTableBytes = (kMaxGroups + 8) * 4;
constexpr int kBarBytes = 256;
// Epilogue staging per warp: a 4 KB 128-byte-swizzled block for GEMM-2's bulk
// stores, or the row-stride-33 layout of its row-by-row path (1024-aligned).
constexpr int kEpiWarp = 5120;
constexpr int kEpiBytes = 4 * kEpiWarp;
constexpr int kSmem = 1024 + kStages * kStageBytes + kTableBytes + kBarBytes + kEpiBytes +
                      kStages * kSfBytes;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kSfCol0 + 8 * kStages <= kTmemCols, "TMEM budget");
static_assert((3 * kStages + 6) * 8 + 8 <= kBarBytes, "barrier area");
static_assert(kTableBytes % 16 == 0 && kEpiBytes % 16 == 0, "scale atoms need 16-byte alignment");

template <int MODE, bool W4>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap map_act,
                           const __grid_constant__ CUtensorMap map_w0,
                           const __grid_constant__ CUtensorMap map_w1,
                           const __grid_constant__ CUtensorMap map_y, const KParams p) {
  constexpr int W_COLS = MODE == 0 ? 64 : 128;  // output columns per tile
  // Transaction bytes of a stage: the A tile, the two B boxes (E2M1 boxes count
  // their packed global bytes, half the shared-memory footprint), the atoms.
  constexpr uint32_t kStageTx = kTileBytes + (W4 ? kTileBytes / 2 : kTileBytes) + kSfBytes;
  constexpr uint32_t kIdescFmt = W4 ? (5u << 10) : 0u;  // B format: E2M1 or E4M3
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* base = smem_raw + pad;
  const uint32_t stage0 = raw_addr + pad;
  // Shared memory: ring | epilogue staging | tile table | barriers | scale atoms.
  float* epi_stage = reinterpret_cast<float*>(base + kStages * kStageBytes);
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + kStages * kStageBytes + kEpiBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes + kEpiBytes + kTableBytes);
  const uint32_t sf_smem0 =
      stage0 + (uint32_t)(kStages * kStageBytes + kEpiBytes + kTableBytes + kBarBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kStages + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
  auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * kStages + 5 + s); };  // scales in TMEM
  const uint32_t sdrain_bar = bar0 + 8u * (3 * kStages + 5);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_wt = (p.N + W_COLS - 1) / W_COLS;
  for (int g = threadIdx.x; g < p.G; g += kThreads) {
    int r0, nr;
    group_rows(p, g, r0, nr);
    tile_start[g] = n_wt * ((nr + 127) / 128);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);  // the producer's arrival carries all the stage's bytes
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < kStages; ++s) mbar_init(sfull_bar(s), 1);
    mbar_init(sdrain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_act);
    prefetch_tensormap(&map_w0);
    prefetch_tensormap(&map_w1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the per-group tile counts
    const int per = (p.G + 31) / 32;
    const int b = lane * per;
    const int e = (b + per < p.G) ? b + per : p.G;
    int local = 0;
    for (int g = b; g < e; ++g) local += tile_start[g];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int g = b; g < e; ++g) {
      const int c = tile_start[g];
      tile_start[g] = run;
      run += c;
    }
    if (lane == 31) tile_start[p.G] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[p.G];
  const int n_k = p.num_kb / 2;  // p.num_kb counts 64-wide slices; a stage holds two

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      Ring rg;
      Armed armed;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile<128>(p, tile_start, tile);
        const int act_row = ti.row0 + ti.tt * 128;
        const int w_row0 = ti.g * p.N + ti.wt * W_COLS;
        const int w_row1 = MODE == 0 ? w_row0 : w_row0 + 64;
        // Atom row blocks: A by token tile, B by 128 rows of the weight atom
        // matrix (GEMM-1: gate/up interleaved per 64 rows; GEMM-2: down).
        const long long a_blk = tile_start[ti.g] / n_wt + ti.tt;
        const long long b_blk = MODE == 0 ? (long long)ti.g * (2 * p.N / 128) + ti.wt
                                          : (long long)ti.g * (p.N / 128) + ti.wt;
        const uint8_t* a_atoms = p.s_act + a_blk * n_k * kAtomBytes;
        const uint8_t* b_atoms = p.s_w0 + b_blk * n_k * kAtomBytes;
        for (int kb = 0; kb < n_k; ++kb) {
          if (!mbar_wait_bounded(empty_bar(rg.s), rg.ph ^ 1u, abort_flag, p.status,
                                 MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(rg.s);
          mbar_arrive_expect_tx(fb, kStageTx);
          const uint32_t st = stage0 + rg.s * kStageBytes;
          const uint32_t sf = sf_smem0 + rg.s * kSfBytes;
          const int kx = kb * kK;
          tma_load_2d(st, &map_act, fb, kx, act_row);
          if (W4) {
            // Tile order: the tile's 128 weight rows (GEMM-1: gate 64 + up 64,
            // half wt & 1 of a 256-row pair block) are one contiguous block.
            const int t = MODE == 0 ? ti.g * (p.N / 128) + ti.wt / 2 : ti.g * (p.N / 128) + ti.wt;
            const int y = MODE == 0 ? (t * n_k + kb) * 256 + (ti.wt & 1) * 128 : (t * n_k + kb) * 128;
            tma_load_2d_hint(st + kTileBytes, &map_w0, fb, 0, y, pol);
          } else {
            tma_load_2d_hint(st + kTileBytes, &map_w0, fb, kx, w_row0, pol);
            tma_load_2d_hint(st + kTileBytes + kTileBytes / 2, &map_w1, fb, kx, w_row1, pol);
          }
          bulk_load_hint(sf, a_atoms + (size_t)kb * kAtomBytes, kAtomBytes, fb, pol);
          bulk_load_hint(sf + kAtomBytes, b_atoms + (size_t)kb * kAtomBytes, kAtomBytes, fb, pol);
          armed.mark(rg);
          rg.next(kStages);
        }
      }
      if (!ok) {
        for (int s = 0; s < kStages; ++s)
          if (armed.mask & (1u << s)) drain_wait(full_bar(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Ring rg;
      bool ok = true, issued = false;
      int local = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t ap = (uint32_t)(local >> 1) & 1u;
        if (!mbar_wait_bounded(tempty_bar(acc), ap ^ 1u, abort_flag, p.status,
                               MOE_DEV_TIMEOUT_MMA, p.limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
        for (int kb = 0; kb < n_k; ++kb) {
          // The scale barrier completes after the stage's data landed and its
          // scales reached TMEM.
          if (!mbar_wait_bounded(sfull_bar(rg.s), rg.ph, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA,
                                 p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = stage0 + rg.s * kStageBytes;
          const uint32_t sf = tmem_base + (uint32_t)(kSfCol0 + 8 * rg.s);
          // +32 bytes along K is +2 in a descriptor's start-address field.
          const uint64_t da = sw128_kmajor_desc(st), db = sw128_kmajor_desc(st + kTileBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            umma_mxf8(d, da + 2 * k, db + 2 * k, idesc_mxf8_e4m3(128, 128, k, k) | kIdescFmt, sf, sf + 4,
                      (kb | k) ? 1u : 0u);
          }
          issued = true;
          umma_commit(empty_bar(rg.s));
          rg.next(kStages);
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
      }
      if (!ok && issued) {
        umma_commit(drain_bar);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else if (warp == kMoverWarp) {
    // ------------------------------------------------------------ scale mover
    if (lane == 0) {
      Ring rg;
      bool ok = true, issued = false;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int kb = 0; kb < n_k; ++kb) {
          if (!mbar_wait_bounded(full_bar(rg.s), rg.ph, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA,
                                 p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tmem_base + (uint32_t)(kSfCol0 + 8 * rg.s);
          tmem_cp_32x128b_warpx4(sf, sf_smem0 + rg.s * kSfBytes);
          tmem_cp_32x128b_warpx4(sf + 4, sf_smem0 + rg.s * kSfBytes + kAtomBytes);
          issued = true;
          umma_commit(sfull_bar(rg.s));
          rg.next(kStages);
        }
      }
      if (!ok && issued) {  // its copies complete before TMEM is freed
        umma_commit(sdrain_bar);
        drain_wait(sdrain_bar, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    float* stg = epi_stage + q * (kEpiWarp / 4);
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t ap = (uint32_t)(local >> 1) & 1u;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull_bar(acc), ap, abort_flag, p.status, MOE_DEV_TIMEOUT_EPILOGUE,
                               p.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = decode_tile<128>(p, tile_start, tile);
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kAccCols);
      const int r = ti.tt * 128 + q * 32 + lane;
      const bool rv = r < ti.nrows;
      if (MODE == 0) {
        // h = silu(gate) * up for columns 0..63 (gate) / 64..127 (up), MXFP8 per 32.
        // Its scale bytes go to the atoms of this token tile (row q*32+lane).
        const long long a_blk = tile_start[ti.g] / n_wt + ti.tt;
        uint8_t* h_atoms = p.out_scale + a_blk * (p.N / 128) * kAtomBytes;
#pragma unroll 1
        for (int c = 0; c < 64; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tb + c, g);
          tmem_ld_32x32b_x32(tb + 64 + c, u);
          tmem_ld_wait();
          const int col = ti.wt * 64 + c;
          if (rv && col < p.N) {
            float hv[32];
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              hv[j] = silu_f(__uint_as_float(g[j])) * __uint_as_float(u[j]);
              amax = fmaxf(amax, fabsf(hv[j]));
            }
            uint32_t w[8];
            int code = 0;
            if (amax == 0.0f) {
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = 0u;
            } else {
              const int sexp = mx_shared_exp(amax);
              code = sexp + 127;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                w[j] = mx_encode(hv[4 * j], sexp) | (mx_encode(hv[4 * j + 1], sexp) << 8) |
                       (mx_encode(hv[4 * j + 2], sexp) << 16) | (mx_encode(hv[4 * j + 3], sexp) << 24);
            }
            const size_t row = (size_t)(ti.row0 + r);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + row * p.N + col);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            h_atoms[(size_t)(col / 128) * kAtomBytes + atom_byte(q * 32 + lane, (col / 32) & 3)] =
                (uint8_t)code;
          }
        }
      } else {
        // fp32 y, 32 x 32 blocks per warp: one TMA bulk store per block from a
        // 128-byte-swizzled buffer when all 32 rows belong to the group, row by
        // row otherwise (a box would also write rows of the next group).
        const int r_first = ti.tt * 128 + q * 32;
        const bool whole = r_first + 32 <= ti.nrows;
        const uint32_t stg_u32 = smem_u32(stg);
        float* y = static_cast<float*>(p.out);
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c, v);
          tmem_ld_wait();
          const int col = ti.wt * 128 + c;
          if (col < p.N) {
            if (lane == 0) bulk_wait_group_read0();  // the last store has read the buffer
            __syncwarp();
            if (whole) {
              uint8_t* rowp = reinterpret_cast<uint8_t*>(stg) + lane * 128;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                    make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&map_y, stg_u32, col, ti.row0 + r_first);
                bulk_commit_group();
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) stg[lane * 33 + j] = __uint_as_float(v[j]);
              __syncwarp();
#pragma unroll 4
              for (int rr = 0; rr < 32; ++rr) {
                const int row = r_first + rr;
                if (row < ti.nrows) y[(size_t)(ti.row0 + row) * p.N + col + lane] = stg[rr * 33 + lane];
              }
              __syncwarp();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
    if (lane == 0) bulk_wait_group0();  // this warp's bulk stores are complete
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int MODE, bool W4>
cudaError_t run_gemm_mx(const GroupedGemmArgs& a, cudaStream_t s) {
  const int Kdim = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const void* act = MODE == 0 ? a.a : a.h;
  const uint8_t* act_scale = MODE == 0 ? a.a_scale : a.h_scale;
  const void* w0 = MODE == 0 ? a.w_gate : a.w_down;
  const void* w1 = MODE == 0 ? a.w_up : a.w_down;
  if (a.rows == 0 || a.G == 0) return cudaSuccess;
  // Whole atoms along K and along the weight rows of a tile.
  if (a.H % 128 || a.I % 128 || a.G > kMaxGroups) return cudaErrorInvalidValue;
  const int G = a.offsets ? a.G : 1;
  CUtensorMap m_act, m_w0, m_w1, m_y;
  bool maps_ok = make_tmap_u8(&m_act, act, Kdim, a.rows, 128);
  if (W4) {  // tile order (moe_tile_mxfp4_weights): GEMM-1 a gate/up pair, GEMM-2 one matrix
    maps_ok = maps_ok && make_tmap_e2m1(&m_w0, w0, (MODE == 0 ? 2ull : 1ull) * G * N * (Kdim / 128), 128);
    m_w1 = m_w0;
  } else {
    maps_ok = maps_ok && make_tmap_u8(&m_w0, w0, Kdim, (uint64_t)G * N, 64) &&
              make_tmap_u8(&m_w1, w1, Kdim, (uint64_t)G * N, 64);
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
  p.s_w0 = MODE == 0 ? a.s_gate : a.s_down;  // weight scale atoms
  p.s_act = act_scale;                       // activation scale atoms, by token tile
  p.out_scale = MODE == 0 ? a.h_scale : nullptr;
  constexpr int W_COLS = MODE == 0 ? 64 : 128;
  const long long n_wt = (N + W_COLS - 1) / W_COLS;
  const long long max_tiles = n_wt * ((a.rows + 127) / 128 + G);
  const int grid = (int)(max_tiles < a.num_sms ? max_tiles : a.num_sms);
  if (MODE == 1) {  // GEMM-2 stores y blocks through a tensor map
    if (!make_tmap_f32_store(&m_y, a.y, (uint64_t)N, (uint64_t)a.rows)) return cudaErrorInvalidValue;
  } else {
    m_y = m_act;  // unused
  }
  grouped_gemm_mx_kernel<MODE, W4><<<grid, kThreads, kSmem, s>>>(m_act, m_w0, m_w1, m_y, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_mx_prepare_device() {
  const cudaError_t errs[] = {
      cudaFuncSetAttribute(grouped_gemm_mx_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  const cudaError_t e = gemm_mx_wide_prepare_device();
  return e != cudaSuccess ? e : gemm_mx_swap_prepare_device();
}

// The tiling of an MX GEMM (mode 0: GEMM-1, 1: GEMM-2): 1 = 128 weight rows
// (this file), 2 = 256 (gemm_mx_wide.cu), 3 = weights as M (gemm_mx_swap.cu).
// Automatic, by rows per expert as the bf16 GEMMs choose: up to 48 on
// average (decode) the weights-as-M tiling, whose MMAs carry no token padding
// (decode shape: MXFP8 GEMM-1 0.358 -> 0.349 ms, 0.99 of HBM); above that 256
// rows for the routed experts (T = 2048: W4A8 GEMM-1 0.64 -> 0.77 of HBM;
// MXFP8 GEMM-1 0.410 -> 0.403 ms, GEMM-2 0.240 -> 0.226 ms), and 128 rows for
// a single group with E4M3 weights (the shared expert), whose 256-row tiles
// would be half as many and leave SMs idle.
int pick_mx_tile(const GroupedGemmArgs& a, int mode) {
  int t = a.mx_tile;
  if (t == 0) {
    const int G = a.offsets ? a.G : 1;
    const double avg_rows = (double)a.rows / (G > 0 ? G : 1);
    t = avg_rows <= 48.0 ? 3 : ((a.w4 || G > 1) ? 2 : 1);
  }
  if (t == 3 && !gemm_mx_swap_supported(a, mode)) t = a.w4 ? 2 : 1;
  if (t == 2 && !gemm_mx_wide_supported(a, mode)) t = 1;
  return t;
}

cudaError_t launch_gemm_mx_gate_up(const GroupedGemmArgs& a, cudaStream_t s) {
  switch (pick_mx_tile(a, 0)) {
    case 3:
      return launch_gemm_mx_swap_gate_up(a, s);
    case 2:
      return launch_gemm_mx_wide_gate_up(a, s);
    default:
      return a.w4 ? run_gemm_mx<0, true>(a, s) : run_gemm_mx<0, false>(a, s);
  }
}

cudaError_t launch_gemm_mx_down(const GroupedGemmArgs& a, cudaStream_t s) {
  switch (pick_mx_tile(a, 1)) {
    case 3:
      return launch_gemm_mx_swap_down(a, s);
    case 2:
      return launch_gemm_mx_wide_down(a, s);
    default:
      return a.w4 ? run_gemm_mx<1, true>(a, s) : run_gemm_mx<1, false>(a, s);
  }
}

}  // namespace moe
