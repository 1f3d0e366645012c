// Step 3: grouped expert GEMM with the SwiGLU epilogue fused, on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM), operands
// staged by TMA. This is the "分组 GMM" / FusedMoEGMM step of the routed path
// ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the
// routed path is the bulk of the MoE block's time) with the expert FFN of
// section 一 (intermediate 1536) in SwiGLU form, bf16 operands. The MXFP8
// form of section 8.2 runs on the block-scaled tensor cores (gemm_mx.cu).
//
//   GEMM-1 (MODE 0):  h[r, i] = silu(sum_c a[r,c] Wg[g,i,c]) * (sum_c a[r,c] Wu[g,i,c])
//   GEMM-2 (MODE 1):  y[r, m] = sum_i h[r,i] Wd[g,m,i]
// for every row r of group g (rows offsets[g] .. offsets[g+1]-1).
//   Gating (MODE 2):  logits[t, e] = sum_c x[t,c] Wr[e,c] for E <= 256, one
//                     group; the epilogue runs the sigmoid top-k routing on
//                     the fp32 accumulators (section 8.5: gating, then routing).
//
// Kernel structure (persistent, one CTA per SM):
//   warp 0      TMA producer (one thread): fills a ring of shared-memory
//               stages, each one K-slice of 64 elements of both operands.
//   warp 1      TMEM allocator + MMA issuer (one thread): tcgen05.mma into a
//               double-buffered TMEM accumulator, tcgen05.commit frees stages.
//   warps 2..5  epilogue: tcgen05.ld the accumulator, SwiGLU / fp32 store.
// Tiles are listed per group on the device (no host read of the group sizes)
// and dealt to CTAs round-robin.
//
// Folded shared expert (optional): group p.fold_group takes its weights from a
// second pair of tensor maps (the shared expert's), so the shared MLP runs as
// one more group of the routed launch instead of on its own stream.
//
// Two tilings (SWAP template flag):
//   SWAP = true   weights are the 128-row MMA operand A (two A tiles: gate and
//                 up rows, or two 128-row blocks of W_down) and BN = 32 tokens
//                 of the group form N. For few tokens per expert (decode) the
//                 kernel is a weight stream and the MMA barely costs anything.
//   SWAP = false  128 tokens form A and 256 weight rows form B with N = 256
//                 (gate 128 + up 128 for GEMM-1), the compute-bound tiling.
//
// Every wait is bounded (about 2 s); on expiry the CTA records an error code
// in the status word, drains its in-flight copies/MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"
#include "gemm_sched.cuh"
#include "ptx.cuh"
#include "topk_key.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;            // K elements per stage = one 128-byte swizzle row of bf16
constexpr int kMaxGroups = 1024;
constexpr int kTopSlots = 8;       // gating epilogue: top-k kept in registers up to this K
constexpr int kMaxSmem = 232448;   // 227 KB dynamic shared memory per CTA

constexpr int kGatherThreads = 128;  // A-row loaders of the gathered GEMM-1: one row each

template <bool SWAP, int MODE, int BN, bool GATHER = false>
struct Geo {
  static constexpr int kTileBytes = 128 * 128;                       // 128 rows x 128 B
  // Gathered GEMM-1: warps 6..9 load the A rows (cp.async) beside the roles below.
  static constexpr int THREADS = GATHER ? 192 + kGatherThreads : 192;
  static constexpr int ACT_ROWS = SWAP ? BN : 128;                   // activation rows / tile
  static constexpr int ACT_BYTES = ACT_ROWS * 128;                   // one 64-wide K slice
  static constexpr int W_BYTES = 2 * kTileBytes;                     // two 128-row weight boxes
  static constexpr int W_COLS = (MODE == 0) ? 128 : 256;             // output cols / tile
  static constexpr int ACC_COLS = SWAP ? 2 * BN : 256;               // TMEM cols / buffer
  static constexpr int TMEM_COLS = (2 * ACC_COLS <= 32) ? 32 : (2 * ACC_COLS <= 64) ? 64
                                   : (2 * ACC_COLS <= 128) ? 128 : (2 * ACC_COLS <= 256) ? 256 : 512;
  static constexpr int TABLE_BYTES = 2 * (kMaxGroups + 8) * 4;  // tile starts, row starts
  static constexpr int BAR_BYTES = 512;
  // Tokens-as-M epilogue: a per-warp 32 x 32 fp32 staging block. GEMM-2 stores
  // it by TMA (4 KB, 128-byte swizzled, 1024-aligned: 5 KB per warp, which also
  // fits the row-stride-33 layout of its row-by-row path); the others use the
  // row-stride-33 layout only.
  static constexpr int EPI_WARP = MODE == 1 ? 5120 : 32 * 33 * 4;
  static constexpr int EPI_BYTES = SWAP ? 0 : 4 * EPI_WARP;
  static constexpr int EXTRA = 1024 + TABLE_BYTES + BAR_BYTES + EPI_BYTES;
  static constexpr int BUDGET = kMaxSmem - EXTRA;
  // One ring whose stages hold both operands of a K slice.
  static constexpr int STAGE_BYTES = ACT_BYTES + W_BYTES;
  static constexpr int ACT_OFF = SWAP ? W_BYTES : 0;                 // within a stage
  static constexpr int W_OFF = SWAP ? 0 : ACT_BYTES;
  static constexpr int S_AB_FREE = BUDGET / STAGE_BYTES;
  static constexpr int S_AB = S_AB_FREE > 8 ? 8 : S_AB_FREE;
  static constexpr int RING_BYTES = S_AB * STAGE_BYTES;
  static constexpr int SMEM = EXTRA + RING_BYTES;
  static constexpr int NBARS = 2 * S_AB + 5;
  static_assert(S_AB >= 2, "shared memory too small for two stages");
  static_assert(ACT_BYTES % 1024 == 0 && W_BYTES % 1024 == 0, "1024-byte alignment of swizzled stages");
  static_assert(EPI_BYTES % 16 == 0, "staging keeps the table aligned");
  static_assert(SMEM <= kMaxSmem, "shared memory budget");
  static_assert(NBARS * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(!SWAP || (BN % 32 == 0 && BN >= 32 && BN <= 128), "token tile");
  static_assert(!GATHER || (!SWAP && MODE == 0), "the gather feeds the tokens-as-M GEMM-1");
};

// Epilogue of one tile: TMEM accumulator (columns tb..) -> h (bf16, SwiGLU),
// y (fp32) or the routing of the gating GEMM. Executed by one warp for its
// 32 lanes.
template <bool SWAP, int MODE, int BN>
__device__ __forceinline__ void epilogue_tile(const KParams& p, const TileInfo& ti, uint32_t tb,
                                              int q, int lane, float* stg, const CUtensorMap* map_y) {
  if (SWAP) {
    // TMEM lane = weight row (output column), TMEM column = token.
    const int r_first = ti.tt * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t v0[32], v1[32];
      tmem_ld_32x32b_x32(tb + c, v0);
      tmem_ld_32x32b_x32(tb + BN + c, v1);
      tmem_ld_wait();
      if (MODE == 0) {
        const int i = ti.wt * 128 + q * 32 + lane;
        __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int r = r_first + c + j;
          const float hv = silu_f(__uint_as_float(v0[j])) * __uint_as_float(v1[j]);
          if (r < ti.nrows && i < p.N) h[(size_t)(ti.row0 + r) * p.N + i] = __float2bfloat16_rn(hv);
        }
      } else {
        const int m0 = ti.wt * 256 + q * 32 + lane, m1 = m0 + 128;
        float* y = static_cast<float*>(p.out);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int r = r_first + c + j;
          if (r < ti.nrows) {
            float* yr = y + (size_t)(ti.row0 + r) * p.N;
            if (m0 < p.N) yr[m0] = __uint_as_float(v0[j]);
            if (m1 < p.N) yr[m1] = __uint_as_float(v1[j]);
          }
        }
      }
    }
  } else {
    // TMEM lane = token row, TMEM column = output column.
    const int r = ti.tt * 128 + q * 32 + lane;
    const bool rv = r < ti.nrows;
    if (MODE == 0) {
      __nv_bfloat16* hrow =
          static_cast<__nv_bfloat16*>(p.out) + (size_t)(ti.row0 + (rv ? r : 0)) * p.N;
#pragma unroll 1
      for (int c = 0; c < 128; c += 32) {
        uint32_t g[32], u[32];
        tmem_ld_32x32b_x32(tb + c, g);
        tmem_ld_32x32b_x32(tb + 128 + c, u);
        tmem_ld_wait();
        const int col = ti.wt * 128 + c;
        if (rv && col < p.N) {
          float hv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) hv[j] = silu_f(__uint_as_float(g[j])) * __uint_as_float(u[j]);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(hv[2 * j], hv[2 * j + 1]);
            pk[j] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(hrow + col);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
    } else if (MODE == 2) {
      // Fused routing of this token: its E logits sit in TMEM columns 0..E-1.
      const int E = p.N;
      const int rbase = ti.row0 + ti.tt * 128 + q * 32;  // this warp's first row
      const int nvalid = ti.nrows - (ti.tt * 128 + q * 32);
      float* lout = static_cast<float*>(p.out);
      const size_t orow = (size_t)(ti.row0 + (rv ? r : 0)) * p.topk;
      if (p.topk <= kTopSlots) {
        // One pass over the logits with the best kTopSlots keys kept sorted
        // in registers (keys are unique, so the order is strict). The logits,
        // when asked for, leave through the warp's 32 x 33 staging block so
        // that each store instruction writes one row's 32 consecutive floats.
        unsigned long long top[kTopSlots];
#pragma unroll
        for (int j = 0; j < kTopSlots; ++j) top[j] = 0ull;
#pragma unroll 1
        for (int c = 0; c < E; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c, v);
          tmem_ld_wait();
          if (lout) {
#pragma unroll
            for (int j = 0; j < 32; ++j) stg[lane * 33 + j] = __uint_as_float(v[j]);
            __syncwarp();
            const int nr = nvalid < 32 ? nvalid : 32;
            for (int rr = 0; rr < nr; ++rr)
              if (c + lane < E) lout[(size_t)(rbase + rr) * E + c + lane] = stg[rr * 33 + lane];
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const unsigned long long key =
                c + j < E ? make_key(__uint_as_float(v[j]), c + j) : 0ull;
#pragma unroll
            for (int s = kTopSlots - 1; s > 0; --s)
              top[s] = key > top[s - 1] ? top[s - 1] : (key > top[s] ? key : top[s]);
            top[0] = key > top[0] ? key : top[0];
          }
        }
        float sig[kTopSlots];
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < kTopSlots; ++k) {
          sig[k] = 1.0f / (1.0f + expf(-key_logit(top[k])));
          if (k < p.topk) sum += sig[k];
        }
        if (rv) {
#pragma unroll
          for (int k = 0; k < kTopSlots; ++k)
            if (k < p.topk) {
              p.topk_idx[orow + k] = key_id(top[k]);
              p.topk_w[orow + k] = (p.route_norm ? sig[k] / sum : sig[k]) * p.scaling;
            }
        }
      } else {
        // K > kTopSlots: K rounds, each taking the largest key below the
        // previous pick, so no list of taken experts is kept.
        float* lrow = lout ? lout + (size_t)(ti.row0 + (rv ? r : 0)) * E : nullptr;
        unsigned long long prev = ~0ull;
        float sum = 0.0f;
#pragma unroll 1
        for (int k = 0; k < p.topk; ++k) {
          unsigned long long best = 0ull;
#pragma unroll 1
          for (int c = 0; c < E; c += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tb + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int e = c + j;
              const float l = __uint_as_float(v[j]);
              if (k == 0 && lrow && rv && e < E) lrow[e] = l;
              const unsigned long long key = e < E ? make_key(l, e) : 0ull;
              if (key < prev && key > best) best = key;
            }
          }
          prev = best;
          const float sig = 1.0f / (1.0f + expf(-key_logit(best)));
          sum += sig;
          if (rv) {
            p.topk_idx[orow + k] = key_id(best);
            p.topk_w[orow + k] = sig;
          }
        }
        if (rv) {
          for (int k = 0; k < p.topk; ++k) {
            const float sig = p.topk_w[orow + k];
            p.topk_w[orow + k] = (p.route_norm ? sig / sum : sig) * p.scaling;
          }
        }
      }
    } else {
      // fp32 y, 32 x 32 blocks per warp. When all 32 rows belong to the group
      // the block leaves by one TMA bulk store from a 128-byte-swizzled 4 KB
      // buffer (16-byte chunk j of row r at chunk j ^ (r % 8)). A block that
      // crosses the group's end goes row by row through the row-stride-33
      // layout, since a TMA box would also write rows of the next group.
      const int r_first = ti.tt * 128 + q * 32;  // this warp's first row in the group
      const bool whole = r_first + 32 <= ti.nrows;
      float* y = static_cast<float*>(p.out);
      const uint32_t stg_u32 = smem_u32(stg);
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c, v);
        tmem_ld_wait();
        const int col = ti.wt * 256 + c;
        if (col < p.N) {  // warp-uniform
          if (lane == 0) bulk_wait_group_read0();  // the last store has read the buffer
          __syncwarp();
          if (whole) {
            uint8_t* row = reinterpret_cast<uint8_t*>(stg) + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(map_y, stg_u32, col, ti.row0 + r_first);
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
  }
}

template <bool SWAP, int MODE, int BN, bool GATHER>
__global__ void __launch_bounds__(Geo<SWAP, MODE, BN, GATHER>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_act,
                        const __grid_constant__ CUtensorMap map_w0,
                        const __grid_constant__ CUtensorMap map_w1,
                        const __grid_constant__ CUtensorMap map_y,
                        const __grid_constant__ CUtensorMap map_w0s,
                        const __grid_constant__ CUtensorMap map_w1s, const KParams p) {
  using Gm = Geo<SWAP, MODE, BN, GATHER>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* base = smem_raw + pad;
  const uint32_t base_u32 = raw_addr + pad;
  // Shared memory: ring | epilogue staging (1024-aligned) | tile table | barriers.
  float* epi_stage = reinterpret_cast<float*>(base + Gm::RING_BYTES);
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + Gm::RING_BYTES + Gm::EPI_BYTES);
  int32_t* row_start = tile_start + kMaxGroups + 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Gm::RING_BYTES + Gm::EPI_BYTES + Gm::TABLE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Gm::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // Barrier slots: full/empty[S_AB], tfull[2], tempty[2], drain.
  constexpr int NS = Gm::S_AB;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NS + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NS + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NS + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NS + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile table: tile_start[g] = tiles of groups before g; row starts.
  const int n_wt = (p.N + Gm::W_COLS - 1) / Gm::W_COLS;
  for (int g = threadIdx.x; g < p.G; g += Gm::THREADS) {
    int r0, nr;
    group_rows(p, g, r0, nr);
    tile_start[g] = n_wt * ((nr + Gm::ACT_ROWS - 1) / Gm::ACT_ROWS);
  }
  fill_row_start(p, row_start, threadIdx.x, Gm::THREADS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      // Gathered: the producer's arrive (weights by TMA) and one asynchronous
      // arrive per loader thread once its copies of the stage have landed.
      mbar_init(full_bar(s), GATHER ? 1 + kGatherThreads : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_act);
    prefetch_tensormap(&map_w0);
    prefetch_tensormap(&map_w1);
    if (p.fold_group >= 0) {
      prefetch_tensormap(&map_w0s);
      prefetch_tensormap(&map_w1s);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Both operands of each 64-wide K slice into one ring stage.
    if (lane == 0) {
      // Weights-as-M streams each weight tile through one CTA: keep it out of
      // the way in L2. Tokens-as-M shares a weight tile among the CTAs of its
      // m-tiles, so it keeps the default policy.
      const uint64_t pol_w = SWAP ? l2_policy_evict_first() : l2_policy_evict_normal();
      Ring rg;
      Armed armed;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile_s<Gm::ACT_ROWS>(p.G, tile_start, row_start, tile);
        const int act_row = ti.row0 + ti.tt * Gm::ACT_ROWS;
        const bool shg = ti.g == p.fold_group;  // the folded shared expert's group
        const CUtensorMap* mw0 = shg ? &map_w0s : &map_w0;
        const CUtensorMap* mw1 = shg ? &map_w1s : &map_w1;
        const int w_row0 = (shg ? 0 : ti.g * p.N) + ti.wt * Gm::W_COLS;
        const int w_row1 = (MODE == 0) ? w_row0 : w_row0 + 128;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(empty_bar(rg.s), rg.ph ^ 1u, abort_flag, p.status,
                                 MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const int kx = kb * kBK;
          const uint32_t fb = full_bar(rg.s);
          mbar_arrive_expect_tx(fb, GATHER ? Gm::W_BYTES : Gm::STAGE_BYTES);
          const uint32_t st = base_u32 + rg.s * Gm::STAGE_BYTES;
          if (!GATHER) tma_load_2d(st + Gm::ACT_OFF, &map_act, fb, kx, act_row);
          if (SWAP) {
            tma_load_2d_hint(st + Gm::W_OFF, mw0, fb, kx, w_row0, pol_w);
            tma_load_2d_hint(st + Gm::W_OFF + Gm::kTileBytes, mw1, fb, kx, w_row1, pol_w);
          } else {
            tma_load_2d(st + Gm::W_OFF, mw0, fb, kx, w_row0);
            tma_load_2d(st + Gm::W_OFF + Gm::kTileBytes, mw1, fb, kx, w_row1);
          }
          armed.mark(rg);
          rg.next(NS);
        }
      }
      if (!ok) {  // let copies already issued land before the CTA exits
        for (int s = 0; s < NS; ++s)
          if (armed.mask & (1u << s)) drain_wait(full_bar(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = SWAP ? idesc_bf16_f32(128, BN) : idesc_bf16_f32(128, 256);
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
        const uint32_t d = tmem_base + (uint32_t)(acc * Gm::ACC_COLS);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(full_bar(rg.s), rg.ph, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA,
                                 p.limit_ns)) {
            ok = false;
            break;
          }
          // Gathered A rows were written by cp.async (the generic proxy); the
          // tensor cores read through the async proxy.
          if (GATHER) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t st = base_u32 + rg.s * Gm::STAGE_BYTES;
          const uint32_t sA = st + (SWAP ? Gm::W_OFF : Gm::ACT_OFF);
          const uint32_t sB = st + (SWAP ? Gm::ACT_OFF : Gm::W_OFF);
          // +32 bytes along K is +2 in a descriptor's start-address field.
          const uint64_t da = sw128_kmajor_desc(sA), db = sw128_kmajor_desc(sB);
          const uint64_t da2 = SWAP ? sw128_kmajor_desc(sA + Gm::kTileBytes) : 0;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kb | k) ? 1u : 0u;
            umma_bf16(d, da + 2 * k, db + 2 * k, kIdesc, accum);
            if (SWAP) umma_bf16(d + BN, da2 + 2 * k, db + 2 * k, kIdesc, accum);
          }
          issued = true;
          umma_commit(empty_bar(rg.s));
          rg.next(NS);
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
      }
      if (!ok && issued) {  // wait for every issued MMA before TMEM is freed
        umma_commit(drain_bar);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else if (GATHER && warp >= 6) {
    // ------------------------------------------------------------ A loader
    // Each loader warp fills 32 of the tile's 128 A rows, four rows per
    // instruction: lane l copies 16-byte chunk c = l % 8 of row 4i + l / 8 of
    // the warp's rows (one 128-byte line per row and stage, so a warp
    // instruction reads four whole lines). A row holds token gather_src[row]
    // / gather_k of x; chunk c lands at position c ^ (row % 8) of the row's
    // 128 bytes (the 128-byte swizzle the MMA descriptors expect). Rows past
    // the group's end are not loaded (their accumulator rows are never
    // stored). Each thread arrives on the stage's full barrier when its
    // copies have landed.
    const int lw = warp - 6;            // loader warp 0..3
    const int c = lane & 7, sub = lane >> 3;
    const uint8_t* x = static_cast<const uint8_t*>(p.gather_x);
    const size_t row_bytes = (size_t)p.num_kb * kBK * 2;
    Ring rg;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile_s<Gm::ACT_ROWS>(p.G, tile_start, row_start, tile);
      const uint8_t* src[8];
      uint32_t off[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rho = lw * 32 + i * 4 + sub;  // row within the tile
        const int r = ti.tt * Gm::ACT_ROWS + rho;
        src[i] = nullptr;
        if (r < ti.nrows) {
          const int f = __ldg(p.gather_src + ti.row0 + r);
          if ((unsigned)f < (unsigned)p.rows) src[i] = x + (size_t)(f / p.gather_k) * row_bytes + c * 16;
        }
        off[i] = (uint32_t)(rho * 128 + ((c ^ (rho & 7)) << 4));
      }
      for (int kb = 0; kb < p.num_kb; ++kb) {
        int go = 1;
        if (lane == 0)
          go = mbar_wait_bounded(empty_bar(rg.s), rg.ph ^ 1u, abort_flag, p.status,
                                 MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, go, 0)) {
          ok = false;
          break;
        }
        const uint32_t dst = base_u32 + rg.s * Gm::STAGE_BYTES + Gm::ACT_OFF;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (src[i]) cp_async_16(dst + off[i], src[i] + (size_t)kb * 128);
        cp_async_arrive_noinc(full_bar(rg.s));
        rg.next(NS);
      }
    }
    cp_async_wait_all();  // this thread's copies have landed before the CTA tears down
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t ap = (uint32_t)(local >> 1) & 1u;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull_bar(acc), ap, abort_flag, p.status,
                               MOE_DEV_TIMEOUT_EPILOGUE, p.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = decode_tile_s<Gm::ACT_ROWS>(p.G, tile_start, row_start, tile);
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * Gm::ACC_COLS);
      epilogue_tile<SWAP, MODE, BN>(p, ti, tb, q, lane, epi_stage + q * (Gm::EPI_WARP / 4), &map_y);
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
    tmem_dealloc(tmem_base, Gm::TMEM_COLS);
  }
}

__global__ void selftest_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    // Nothing arrives on this barrier: the wait must give up on its own.
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, MOE_DEV_TIMEOUT_SELFTEST,
                      limit_ns);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

// 2-D tensor [outer, inner] (inner contiguous), box {128 bytes of K,
// box_rows}, 128-byte swizzle, zero fill out of range: 64 bf16 or 128 E4M3
// bytes, the MMA operand layout of either.
bool make_map(CUtensorMap* m, const void* ptr, bool fp8, uint64_t inner, uint64_t outer,
              uint32_t box_rows) {
  if (!g_encode) return false;
  const uint64_t esize = fp8 ? 1 : 2;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {(cuuint32_t)(fp8 ? 2 * kBK : kBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                              const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D fp32 tensor [outer, inner], box {32, 32} (128-byte rows), 128-byte
// swizzle: the staging block of the GEMM-2 epilogue's bulk stores.
bool make_map_f32(CUtensorMap* m, void* ptr, uint64_t inner, uint64_t outer) {
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool make_tmap_f32_store(CUtensorMap* m, void* ptr, uint64_t inner, uint64_t outer) {
  return make_map_f32(m, ptr, inner, outer);
}

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  return make_map(m, ptr, false, inner, outer, box_rows);
}

bool make_tmap_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  return make_map(m, ptr, true, inner, outer, box_rows);
}

bool make_tmap_e2m1(CUtensorMap* m, const void* ptr, uint64_t rows64, uint32_t box_rows) {
  if (!g_encode || box_rows == 0 || box_rows > 256 || (reinterpret_cast<uintptr_t>(ptr) & 31)) return false;
  const cuuint64_t dims[2] = {128, rows64};
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(ptr), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <bool SWAP, int MODE, int BN, bool GATHER = false>
cudaError_t run_gemm(const GroupedGemmArgs& a, cudaStream_t s) {
  using Gm = Geo<SWAP, MODE, BN, GATHER>;
  const int Kdim = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const void* act = MODE == 0 ? a.a : a.h;
  const void* w0 = MODE == 0 ? a.w_gate : a.w_down;
  const void* w1 = MODE == 0 ? a.w_up : a.w_down;
  if (a.rows == 0 || a.G == 0) return cudaSuccess;
  const int G = a.offsets ? a.G : 1;
  // A folded shared expert is the last group; its weights have their own maps.
  const bool fold = a.shared_w_gate != nullptr && a.offsets != nullptr;
  const int Gw = fold ? G - 1 : G;  // groups whose weights are in w0 / w1
  CUtensorMap m_act, m_w0, m_w1, m_y, m_w0s, m_w1s;
  if ((!GATHER && !make_map(&m_act, act, false, Kdim, a.rows, Gm::ACT_ROWS)) ||
      !make_map(&m_w0, w0, false, Kdim, (uint64_t)Gw * N, 128) ||
      !make_map(&m_w1, w1, false, Kdim, (uint64_t)Gw * N, 128))
    return cudaErrorInvalidValue;
  if (GATHER) m_act = m_w0;  // unused: the A rows are gathered
  if (fold) {
    const void* s0 = MODE == 0 ? a.shared_w_gate : a.shared_w_down;
    const void* s1 = MODE == 0 ? a.shared_w_up : a.shared_w_down;
    if (!make_map(&m_w0s, s0, false, Kdim, (uint64_t)N, 128) ||
        !make_map(&m_w1s, s1, false, Kdim, (uint64_t)N, 128))
      return cudaErrorInvalidValue;
  } else {
    m_w0s = m_w0;  // unused
    m_w1s = m_w1;
  }
  auto kern = grouped_gemm_kernel<SWAP, MODE, BN, GATHER>;
  KParams p = {};
  p.offsets = a.offsets;
  p.G = G;
  p.rows = a.rows;
  p.num_kb = (Kdim + kBK - 1) / kBK;
  p.N = N;
  p.out = MODE == 0 ? a.h : static_cast<void*>(a.y);
  p.status = a.status;
  p.limit_ns = a.wait_limit_ns;
  p.topk_idx = a.topk_idx;
  p.topk_w = a.topk_w;
  p.topk = a.topk;
  p.scaling = a.scaling;
  p.route_norm = a.route_norm;
  p.fold_group = fold ? G - 1 : -1;
  p.gather_src = GATHER ? a.gather_src : nullptr;
  p.gather_k = a.gather_k;
  p.gather_x = a.gather_x;
  const long long n_wt = (N + Gm::W_COLS - 1) / Gm::W_COLS;
  const long long max_tiles = n_wt * ((a.rows + Gm::ACT_ROWS - 1) / Gm::ACT_ROWS + G);
  const int grid = (int)(max_tiles < a.num_sms ? max_tiles : a.num_sms);
  // GEMM-2 tokens-as-M stores y through a tensor map; elsewhere the slot is unused.
  if (MODE == 1 && !SWAP) {
    if (!make_map_f32(&m_y, a.y, (uint64_t)N, (uint64_t)a.rows)) return cudaErrorInvalidValue;
  } else {
    m_y = m_act;
  }
  kern<<<grid, Gm::THREADS, Gm::SMEM, s>>>(m_act, m_w0, m_w1, m_y, m_w0s, m_w1s, p);
  return cudaGetLastError();
}

template <bool SWAP, int MODE, int BN, bool GATHER = false>
cudaError_t set_smem_attribute() {
  return cudaFuncSetAttribute(grouped_gemm_kernel<SWAP, MODE, BN, GATHER>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Geo<SWAP, MODE, BN, GATHER>::SMEM);
}

int pick_mode(const GroupedGemmArgs& a) {
  int m = a.mode;
  if (m != kModeWeightsM && m != kModeTokensM && m != kModePair) {
    const int G = a.offsets ? a.G : 1;
    const double avg_rows = (double)a.rows / (G > 0 ? G : 1);
    m = avg_rows <= 48.0 ? kModeWeightsM : kModeTokensM;
  }
  if (m == kModePair && !gemm_pair_supported(a)) m = kModeTokensM;
  return m;
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemmArgs& a, cudaStream_t s) {
  switch (pick_mode(a)) {
    case kModeWeightsM:
      return run_gemm<true, MODE, 32>(a, s);
    case kModePair:
      return MODE == 0 ? launch_gemm_pair_gate_up(a, s) : launch_gemm_pair_down(a, s);
    default:
      if (MODE == 0 && a.gather_src) return run_gemm<false, 0, 32, true>(a, s);
      return run_gemm<false, MODE, 32>(a, s);
  }
}

}  // namespace

bool gemm_init_driver() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode != nullptr;
}

cudaError_t gemm_prepare_device() {
  const cudaError_t errs[] = {
      set_smem_attribute<true, 0, 32>(), set_smem_attribute<false, 0, 32>(),
      set_smem_attribute<true, 1, 32>(), set_smem_attribute<false, 1, 32>(),
      set_smem_attribute<false, 2, 32>(), set_smem_attribute<false, 0, 32, true>(),
      gemm_pair_prepare_device()};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

int gemm_pick_mode(const GroupedGemmArgs& a) { return pick_mode(a); }

cudaError_t launch_gemm_gate_up(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_mode<0>(a, s);
}

cudaError_t launch_gemm_down(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_mode<1>(a, s);
}

cudaError_t launch_gate_route(const GroupedGemmArgs& a, cudaStream_t s) {
  // MODE 2 reads the MODE 1 operand slots: act = a.h (x), K = a.I (hidden),
  // N = a.H (experts), weights = a.w_down (router).
  return run_gemm<false, 2, 32>(a, s);
}

cudaError_t launch_selftest_wait(int* status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
