// Step 3: grouped expert GEMM with the SwiGLU epilogue fused, on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM), operands
// staged by TMA. This is the "分组 GMM" / FusedMoEGMM step of the routed path
// ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the
// routed path is the bulk of the MoE block's time) with the expert FFN of
// section 一 (intermediate 1536) in SwiGLU form, and the MXFP8 weights of
// section 8.2 (W8A8, E4M3 elements with one E8M0 scale per 32 along K).
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
// With MXFP8 weights (WQ) two more roles run:
//   warps 6..9  converters: expand each E4M3 weight slice (staged by TMA in a
//               deeper ring of raw bytes) times its E8M0 block scale into the
//               swizzled bf16 operand layout. The expansion is exact, so the
//               bf16 MMA with fp32 accumulation computes the MX product.
//   warp 10     activation TMA producer, so the deep weight ring never waits
//               on the shallow bf16 ring; warp 0 then only streams weights.
// Tiles are listed per group on the device (no host read of the group sizes)
// and dealt to CTAs round-robin.
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
#include "mx.cuh"
#include "gemm_sched.cuh"
#include "ptx.cuh"
#include "topk_key.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;            // K elements per stage = one 128-byte swizzle row of bf16
constexpr int kMaxGroups = 1024;
constexpr int kMaxSmem = 232448;   // 227 KB dynamic shared memory per CTA
constexpr int kConvWarp0 = 6;      // first converter warp (WQ)
constexpr int kConvWarps = 16;     // converter warps (WQ): four per SM sub-partition
constexpr int kActWarp = kConvWarp0 + kConvWarps;  // activation producer warp (WQ)

template <bool SWAP, int MODE, int BN, bool WQ>
struct Geo {
  static constexpr int kTileBytes = 128 * 128;                       // 128 rows x 128 B
  static constexpr int THREADS = WQ ? (kActWarp + 1) * 32 : 192;
  static constexpr int ACT_ROWS = SWAP ? BN : 128;                   // activation rows / tile
  static constexpr int ACT_BYTES = ACT_ROWS * 128;                   // one 64-wide K slice
  static constexpr int W_BYTES = 2 * kTileBytes;                     // two 128-row weight boxes
  static constexpr int W_COLS = (MODE == 0) ? 128 : 256;             // output cols / tile
  static constexpr int ACC_COLS = SWAP ? 2 * BN : 256;               // TMEM cols / buffer
  static constexpr int TMEM_COLS = (2 * ACC_COLS <= 32) ? 32 : (2 * ACC_COLS <= 64) ? 64
                                   : (2 * ACC_COLS <= 128) ? 128 : (2 * ACC_COLS <= 256) ? 256 : 512;
  static constexpr int TABLE_BYTES = (kMaxGroups + 8) * 4;
  static constexpr int BAR_BYTES = 512;
  // Tokens-as-M epilogue: per-warp 32 x 32 fp32 staging (row stride 33) so
  // output rows leave as contiguous 128-byte stores.
  static constexpr int EPI_BYTES = SWAP ? 0 : 4 * 32 * 33 * 4;
  static constexpr int EXTRA = 1024 + TABLE_BYTES + BAR_BYTES + EPI_BYTES;
  static constexpr int BUDGET = kMaxSmem - EXTRA;
  // bf16 weights: one ring whose stages hold both operands of a K slice.
  static constexpr int STAGE_BYTES = ACT_BYTES + W_BYTES;
  static constexpr int ACT_OFF = SWAP ? W_BYTES : 0;                 // within a combined stage
  static constexpr int W_OFF = SWAP ? 0 : ACT_BYTES;
  static constexpr int S_AB_FREE = BUDGET / STAGE_BYTES;
  static constexpr int S_AB = WQ ? 0 : (S_AB_FREE > 8 ? 8 : S_AB_FREE);
  // MXFP8 weights: three rings. Raw E4M3 weight slices (deep, streamed from
  // HBM), converted bf16 weight slices (shallow), activation slices (deep).
  static constexpr int RAW_K = 2 * kBK;                              // fp8 K per raw stage (two slices)
  static constexpr int RAW_BYTES = 2 * 128 * RAW_K;                  // two fp8 boxes of 128 x 128
  static constexpr int S_W = WQ ? 3 : 0;
  static constexpr int S_ACT = WQ ? (SWAP ? 8 : 2) : 0;
  static constexpr int S_RAW_FREE = WQ ? (BUDGET - S_W * W_BYTES - S_ACT * ACT_BYTES) / RAW_BYTES : 0;
  static constexpr int S_RAW = S_RAW_FREE > 8 ? 8 : S_RAW_FREE;
  static constexpr int RING_BYTES = WQ ? S_W * W_BYTES + S_ACT * ACT_BYTES + S_RAW * RAW_BYTES
                                       : S_AB * STAGE_BYTES;
  static constexpr int SMEM = EXTRA + RING_BYTES;
  static constexpr int NBARS = WQ ? 2 * (S_W + S_ACT + S_RAW) + 5 : 2 * S_AB + 5;
  static_assert(WQ || S_AB >= 2, "shared memory too small for two stages");
  static_assert(!WQ || S_RAW >= 2, "shared memory too small for the raw weight ring");
  static_assert(ACT_BYTES % 1024 == 0 && W_BYTES % 1024 == 0 && RAW_BYTES % 1024 == 0,
                "1024-byte alignment of swizzled stages");
  static_assert(SMEM <= kMaxSmem, "shared memory budget");
  static_assert(NBARS * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(!SWAP || (BN % 32 == 0 && BN >= 32 && BN <= 128), "token tile");
};

// Epilogue of one tile: TMEM accumulator (columns tb..) -> h (bf16, SwiGLU,
// MX-rounded when MXH) or y (fp32). Executed by one warp for its 32 lanes.
template <bool SWAP, int MODE, int BN, bool MXH>
__device__ __forceinline__ void epilogue_tile(const KParams& p, const TileInfo& ti, uint32_t tb,
                                              int q, int lane, float* stg) {
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
          float hv = silu_f(__uint_as_float(v0[j])) * __uint_as_float(v1[j]);
          if (MXH) {  // MX block of 32 along I = this warp's 32 lanes
            float amax = fabsf(hv);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
              amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
            hv = mx_roundtrip(hv, amax);
          }
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
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            hv[j] = silu_f(__uint_as_float(g[j])) * __uint_as_float(u[j]);
            amax = fmaxf(amax, fabsf(hv[j]));
          }
          if (MXH) {  // MX block of 32 along I = this thread's 32 columns
#pragma unroll
            for (int j = 0; j < 32; ++j) hv[j] = mx_roundtrip(hv[j], amax);
          }
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
      // Round k takes the largest key below the previous pick (keys are
      // unique), so no list of taken experts is kept.
      const int E = p.N;
      float* lrow = static_cast<float*>(p.out);
      if (lrow) lrow += (size_t)(ti.row0 + (rv ? r : 0)) * E;
      const size_t orow = (size_t)(ti.row0 + (rv ? r : 0)) * p.topk;
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
    } else {
      // fp32 y: each 32 x 32 block goes through the warp's staging tile so
      // that every store instruction writes 128 contiguous bytes of one row.
      const int r_first = ti.tt * 128 + q * 32;  // this warp's first row in the group
      float* y = static_cast<float*>(p.out);
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tb + c, v);
        tmem_ld_wait();
        const int col = ti.wt * 256 + c;
        if (col < p.N) {  // warp-uniform
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

template <bool SWAP, int MODE, int BN, bool WQ>
__global__ void __launch_bounds__(Geo<SWAP, MODE, BN, WQ>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_act,
                        const __grid_constant__ CUtensorMap map_w0,
                        const __grid_constant__ CUtensorMap map_w1, const KParams p) {
  using Gm = Geo<SWAP, MODE, BN, WQ>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* base = smem_raw + pad;
  const uint32_t base_u32 = raw_addr + pad;
  // Ring regions (WQ: converted weights, activations, raw fp8; else combined).
  const uint32_t w_ring = base_u32;                                  // WQ
  const uint32_t act_ring = base_u32 + Gm::S_W * Gm::W_BYTES;        // WQ
  const uint32_t raw_ring = act_ring + Gm::S_ACT * Gm::ACT_BYTES;    // WQ
  uint8_t* w_ring_p = base;
  const uint8_t* raw_ring_p = base + (raw_ring - base_u32);
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + Gm::RING_BYTES);
  float* epi_stage = reinterpret_cast<float*>(base + Gm::RING_BYTES + Gm::TABLE_BYTES + Gm::BAR_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Gm::RING_BYTES + Gm::TABLE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Gm::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // Barrier slots. bf16: full/empty[S_AB]. WQ: wfull/wempty[S_W], afull/aempty[S_ACT],
  // rfull/rempty[S_RAW]. Both: tfull[2], tempty[2], drain.
  constexpr int NS1 = WQ ? Gm::S_W : Gm::S_AB;  // "full/empty" = combined or converted-weight ring
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NS1 + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NS1 + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NS1 + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NS1 + 4);
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * NS1 + 5 + s); };
  auto aempty_bar = [&](int s) { return bar0 + 8u * (2 * NS1 + 5 + Gm::S_ACT + s); };
  auto rfull_bar = [&](int s) { return bar0 + 8u * (2 * NS1 + 5 + 2 * Gm::S_ACT + s); };
  auto rempty_bar = [&](int s) { return bar0 + 8u * (2 * NS1 + 5 + 2 * Gm::S_ACT + Gm::S_RAW + s); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile table: tile_start[g] = tiles of groups before g.
  const int n_wt = (p.N + Gm::W_COLS - 1) / Gm::W_COLS;
  for (int g = threadIdx.x; g < p.G; g += Gm::THREADS) {
    int r0, nr;
    group_rows(p, g, r0, nr);
    tile_start[g] = n_wt * ((nr + Gm::ACT_ROWS - 1) / Gm::ACT_ROWS);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS1; ++s) {
      mbar_init(full_bar(s), WQ ? kConvWarps : 1);  // WQ: one arrival per converter warp
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < Gm::S_ACT; ++s) {
      mbar_init(afull_bar(s), 1);
      mbar_init(aempty_bar(s), 1);
    }
    for (int s = 0; s < Gm::S_RAW; ++s) {
      mbar_init(rfull_bar(s), 1);
      mbar_init(rempty_bar(s), kConvWarps);
    }
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
    // bf16: both operands of each K slice into the combined ring.
    // WQ: only the fp8 weight boxes, into the raw ring.
    if (lane == 0) {
      // Weights-as-M streams each weight tile through one CTA: keep it out of
      // the way in L2. Tokens-as-M shares a weight tile among the CTAs of its
      // m-tiles, so it keeps the default policy.
      const uint64_t pol_w = SWAP ? l2_policy_evict_first() : l2_policy_evict_normal();
      constexpr int RING = WQ ? Gm::S_RAW : Gm::S_AB;
      Ring rg;
      Armed armed;
      bool ok = true;
      // bf16: one combined stage per 64-wide K slice. WQ: one raw stage per two slices.
      const int n_steps = WQ ? (p.num_kb + 1) / 2 : p.num_kb;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile<Gm::ACT_ROWS>(p, tile_start, tile);
        const int act_row = ti.row0 + ti.tt * Gm::ACT_ROWS;
        const int w_row0 = ti.g * p.N + ti.wt * Gm::W_COLS;
        const int w_row1 = (MODE == 0) ? w_row0 : w_row0 + 128;
        for (int kb = 0; kb < n_steps; ++kb) {
          const uint32_t eb = WQ ? rempty_bar(rg.s) : empty_bar(rg.s);
          if (!mbar_wait_bounded(eb, rg.ph ^ 1u, abort_flag, p.status, MOE_DEV_TIMEOUT_PRODUCER,
                                 p.limit_ns)) {
            ok = false;
            break;
          }
          if (WQ) {
            const int kx = kb * Gm::RAW_K;
            const uint32_t fb = rfull_bar(rg.s);
            mbar_arrive_expect_tx(fb, Gm::RAW_BYTES);
            const uint32_t r = raw_ring + rg.s * Gm::RAW_BYTES;
            tma_load_2d_hint(r, &map_w0, fb, kx, w_row0, pol_w);
            tma_load_2d_hint(r + Gm::RAW_BYTES / 2, &map_w1, fb, kx, w_row1, pol_w);
          } else {
            const int kx = kb * kBK;
            const uint32_t fb = full_bar(rg.s);
            mbar_arrive_expect_tx(fb, Gm::STAGE_BYTES);
            const uint32_t st = base_u32 + rg.s * Gm::STAGE_BYTES;
            tma_load_2d(st + Gm::ACT_OFF, &map_act, fb, kx, act_row);
            if (SWAP) {
              tma_load_2d_hint(st + Gm::W_OFF, &map_w0, fb, kx, w_row0, pol_w);
              tma_load_2d_hint(st + Gm::W_OFF + Gm::kTileBytes, &map_w1, fb, kx, w_row1, pol_w);
            } else {
              tma_load_2d(st + Gm::W_OFF, &map_w0, fb, kx, w_row0);
              tma_load_2d(st + Gm::W_OFF + Gm::kTileBytes, &map_w1, fb, kx, w_row1);
            }
          }
          armed.mark(rg);
          rg.next(RING);
        }
      }
      if (!ok) {  // let copies already issued land before the CTA exits
        for (int s = 0; s < RING; ++s)
          if (armed.mask & (1u << s))
            drain_wait(WQ ? rfull_bar(s) : full_bar(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = SWAP ? idesc_bf16_f32(128, BN) : idesc_bf16_f32(128, 256);
      Ring rw, ra;  // combined (or converted-weight) ring; activation ring (WQ)
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
          bool got = mbar_wait_bounded(full_bar(rw.s), rw.ph, abort_flag, p.status,
                                       MOE_DEV_TIMEOUT_MMA, p.limit_ns);
          if (WQ && got)
            got = mbar_wait_bounded(afull_bar(ra.s), ra.ph, abort_flag, p.status,
                                    MOE_DEV_TIMEOUT_MMA, p.limit_ns);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sW, sAct;
          if (WQ) {
            sW = w_ring + rw.s * Gm::W_BYTES;
            sAct = act_ring + ra.s * Gm::ACT_BYTES;
          } else {
            const uint32_t st = base_u32 + rw.s * Gm::STAGE_BYTES;
            sW = st + Gm::W_OFF;
            sAct = st + Gm::ACT_OFF;
          }
          const uint32_t sA = SWAP ? sW : sAct;
          const uint32_t sB = SWAP ? sAct : sW;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kb | k) ? 1u : 0u;
            const uint64_t bdesc = sw128_kmajor_desc(sB + k * 32);
            umma_bf16(d, sw128_kmajor_desc(sA + k * 32), bdesc, kIdesc, accum);
            if (SWAP)
              umma_bf16(d + BN, sw128_kmajor_desc(sA + Gm::kTileBytes + k * 32), bdesc, kIdesc,
                        accum);
          }
          issued = true;
          umma_commit(empty_bar(rw.s));
          rw.next(NS1);
          if (WQ) {
            umma_commit(aempty_bar(ra.s));
            ra.next(Gm::S_ACT);
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
      }
      if (!ok && issued) {  // wait for every issued MMA before TMEM is freed
        umma_commit(drain_bar);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else if (warp < kConvWarp0) {
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
      const TileInfo ti = decode_tile<Gm::ACT_ROWS>(p, tile_start, tile);
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * Gm::ACC_COLS);
      epilogue_tile<SWAP, MODE, BN, WQ>(p, ti, tb, q, lane, epi_stage + q * 32 * 33);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  } else if (WQ && warp < kActWarp) {
    // ------------------------------------------------------------ converters (WQ)
    // A raw stage holds 128 K-bytes (two MMA slices) of the 256 weight rows,
    // 128-byte swizzled. Thread ct owns logical 16-byte chunk q of each
    // slice for rows (ct & 7) + 8 (ct >> 5) + kRowStep j, so the 8 lanes of
    // every shared-memory phase touch 8 different rows: conflict-free reads
    // of the raw rows and writes of the bf16 rows. The E8M0 scales of the
    // next raw stage (4 blocks per row) are loaded while this one converts.
    constexpr int kRowStep = 8 * kConvWarps;
    constexpr int kRowsPer = 256 / kRowStep;
    const int ct = threadIdx.x - kConvWarp0 * 32;
    const int q = (ct >> 3) & 3;
    const int row_base = (ct & 7) + 8 * (ct >> 5);
    const int n_raw = (p.num_kb + 1) / 2;
    auto load_scales = [&](uint32_t (&sw)[kRowsPer], int w_row0, int w_row1, int kr) {
#pragma unroll
      for (int j = 0; j < kRowsPer; ++j) {
        const int row = row_base + kRowStep * j;
        const int box = row >> 7;
        const int grow = (box ? w_row1 : w_row0) + (row & 127);
        const uint8_t* sp = (box ? p.s_w1 : p.s_w0) + (size_t)grow * p.sstride + 4 * kr;
        uint32_t v = 0x7F7F7F7Fu;
        if (grow < p.w_rows) {
          if ((p.sstride & 3) == 0) {
            v = __ldg(reinterpret_cast<const uint32_t*>(sp));
          } else {
            v = 0;
            for (int b = 0; b < 4; ++b)
              v |= (uint32_t)((4 * kr + b < p.sstride) ? __ldg(sp + b) : 127) << (8 * b);
          }
        }
        sw[j] = v;
      }
    };
    auto weight_rows = [&](int tile, int& w_row0, int& w_row1) {
      const TileInfo ti = decode_tile<Gm::ACT_ROWS>(p, tile_start, tile);
      w_row0 = ti.g * p.N + ti.wt * Gm::W_COLS;
      w_row1 = (MODE == 0) ? w_row0 : w_row0 + 128;
    };
    Ring rw, rr;
    int tile = blockIdx.x, kr = 0, w_row0 = 0, w_row1 = 0;
    uint32_t sw[kRowsPer], sw_next[kRowsPer];
    if (tile < total) {
      weight_rows(tile, w_row0, w_row1);
      load_scales(sw, w_row0, w_row1, 0);
    }
    bool ok = true;
    while (ok && tile < total) {
      int ntile = tile, nkr = kr + 1, nw0 = w_row0, nw1 = w_row1;
      if (nkr == n_raw) {
        ntile += gridDim.x;
        nkr = 0;
        if (ntile < total) weight_rows(ntile, nw0, nw1);
      }
      if (ntile < total) load_scales(sw_next, nw0, nw1, nkr);
      int ok1 = 1;
      if (lane == 0)
        ok1 = mbar_wait_bounded(rfull_bar(rr.s), rr.ph, abort_flag, p.status,
                                MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns);
      ok1 = __shfl_sync(0xFFFFFFFFu, ok1, 0);
      if (!ok1) break;
      const uint8_t* rsrc = raw_ring_p + rr.s * Gm::RAW_BYTES;
      for (int half = 0; half < 2 && 2 * kr + half < p.num_kb; ++half) {
        if (lane == 0)
          ok1 = mbar_wait_bounded(empty_bar(rw.s), rw.ph ^ 1u, abort_flag, p.status,
                                  MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns);
        ok1 = __shfl_sync(0xFFFFFFFFu, ok1, 0);
        if (!ok1) {
          ok = false;
          break;
        }
        uint8_t* dst = w_ring_p + rw.s * Gm::W_BYTES;
        const int c = q + 4 * half;  // logical 16-byte chunk of the 128-byte raw row
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j) {
          const int row = row_base + kRowStep * j;
          const int box = row >> 7, r = row & 127;
          const uint4 raw = *reinterpret_cast<const uint4*>(rsrc + box * Gm::kTileBytes + r * 128 +
                                                            ((c ^ (r & 7)) << 4));
          const int sc = (int)((sw[j] >> (8 * (2 * half + (q >> 1)))) & 0xFFu);
          uint8_t* drow = dst + box * Gm::kTileBytes + r * 128;
          e4m3x16_to_bf16_store(raw, sc, reinterpret_cast<uint4*>(drow + (((2 * q) ^ (r & 7)) << 4)),
                                reinterpret_cast<uint4*>(drow + (((2 * q + 1) ^ (r & 7)) << 4)));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full_bar(rw.s));
        rw.next(NS1);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty_bar(rr.s));
      rr.next(Gm::S_RAW);
#pragma unroll
      for (int j = 0; j < kRowsPer; ++j) sw[j] = sw_next[j];
      tile = ntile;
      kr = nkr;
      w_row0 = nw0;
      w_row1 = nw1;
    }
  } else if (WQ && warp == kActWarp) {
    // ------------------------------------------------------------ activation producer (WQ)
    if (lane == 0) {
      Ring ra;
      Armed armed;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile<Gm::ACT_ROWS>(p, tile_start, tile);
        const int act_row = ti.row0 + ti.tt * Gm::ACT_ROWS;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(aempty_bar(ra.s), ra.ph ^ 1u, abort_flag, p.status,
                                 MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = afull_bar(ra.s);
          mbar_arrive_expect_tx(fb, Gm::ACT_BYTES);
          tma_load_2d(act_ring + ra.s * Gm::ACT_BYTES, &map_act, fb, kb * kBK, act_row);
          armed.mark(ra);
          ra.next(Gm::S_ACT);
        }
      }
      if (!ok) {
        for (int s = 0; s < Gm::S_ACT; ++s)
          if (armed.mask & (1u << s)) drain_wait(afull_bar(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
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
// box_rows}, 128-byte swizzle, zero fill out of range: 64 bf16 (the MMA
// operand layout) or 128 fp8 weight bytes (the converters' source).
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

}  // namespace

bool make_tmap_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  return make_map(m, ptr, true, inner, outer, box_rows);
}

namespace {

template <bool SWAP, int MODE, int BN, bool WQ>
cudaError_t run_gemm(const GroupedGemmArgs& a, cudaStream_t s) {
  using Gm = Geo<SWAP, MODE, BN, WQ>;
  const int Kdim = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const void* act = MODE == 0 ? a.a : a.h;
  const void* w0 = MODE == 0 ? a.w_gate : a.w_down;
  const void* w1 = MODE == 0 ? a.w_up : a.w_down;
  if (a.rows == 0 || a.G == 0) return cudaSuccess;
  const int G = a.offsets ? a.G : 1;
  CUtensorMap m_act, m_w0, m_w1;
  if (!make_map(&m_act, act, false, Kdim, a.rows, Gm::ACT_ROWS) ||
      !make_map(&m_w0, w0, WQ, Kdim, (uint64_t)G * N, 128) ||
      !make_map(&m_w1, w1, WQ, Kdim, (uint64_t)G * N, 128))
    return cudaErrorInvalidValue;
  auto kern = grouped_gemm_kernel<SWAP, MODE, BN, WQ>;
  KParams p;
  p.offsets = a.offsets;
  p.G = G;
  p.rows = a.rows;
  p.num_kb = (Kdim + kBK - 1) / kBK;
  p.N = N;
  p.out = MODE == 0 ? a.h : static_cast<void*>(a.y);
  p.status = a.status;
  p.limit_ns = a.wait_limit_ns;
  p.s_w0 = MODE == 0 ? a.s_gate : a.s_down;
  p.s_w1 = MODE == 0 ? a.s_up : a.s_down;
  p.sstride = Kdim / 32;
  p.w_rows = G * N;
  p.topk_idx = a.topk_idx;
  p.topk_w = a.topk_w;
  p.topk = a.topk;
  p.scaling = a.scaling;
  p.route_norm = a.route_norm;
  const long long n_wt = (N + Gm::W_COLS - 1) / Gm::W_COLS;
  const long long max_tiles = n_wt * ((a.rows + Gm::ACT_ROWS - 1) / Gm::ACT_ROWS + G);
  const int grid = (int)(max_tiles < a.num_sms ? max_tiles : a.num_sms);
  kern<<<grid, Gm::THREADS, Gm::SMEM, s>>>(m_act, m_w0, m_w1, p);
  return cudaGetLastError();
}

template <bool SWAP, int MODE, int BN, bool WQ>
cudaError_t set_smem_attribute() {
  return cudaFuncSetAttribute(grouped_gemm_kernel<SWAP, MODE, BN, WQ>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<SWAP, MODE, BN, WQ>::SMEM);
}

int pick_mode(const GroupedGemmArgs& a) {
  if (a.mode == kModeWeightsM || a.mode == kModeTokensM) return a.mode;
  const int G = a.offsets ? a.G : 1;
  const double avg_rows = (double)a.rows / (G > 0 ? G : 1);
  return avg_rows <= 48.0 ? kModeWeightsM : kModeTokensM;
}

template <int MODE>
cudaError_t launch_mode(const GroupedGemmArgs& a, cudaStream_t s) {
  const bool swap = pick_mode(a) == kModeWeightsM;
  if (a.mx) return swap ? run_gemm<true, MODE, 32, true>(a, s) : run_gemm<false, MODE, 32, true>(a, s);
  return swap ? run_gemm<true, MODE, 32, false>(a, s) : run_gemm<false, MODE, 32, false>(a, s);
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
      set_smem_attribute<true, 0, 32, false>(), set_smem_attribute<false, 0, 32, false>(),
      set_smem_attribute<true, 1, 32, false>(), set_smem_attribute<false, 1, 32, false>(),
      set_smem_attribute<true, 0, 32, true>(),  set_smem_attribute<false, 0, 32, true>(),
      set_smem_attribute<true, 1, 32, true>(),  set_smem_attribute<false, 1, 32, true>(),
      set_smem_attribute<false, 2, 32, false>()};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_gemm_gate_up(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_mode<0>(a, s);
}

cudaError_t launch_gemm_down(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_mode<1>(a, s);
}

cudaError_t launch_gate_route(const GroupedGemmArgs& a, cudaStream_t s) {
  // MODE 2 reads the MODE 1 operand slots: act = a.h (x), K = a.I (hidden),
  // N = a.H (experts), weights = a.w_down (router).
  return run_gemm<false, 2, 32, false>(a, s);
}

cudaError_t launch_selftest_wait(int* status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
