// Step 3 on CTA pairs: the grouped expert GEMM (GEMM-1 with the SwiGLU
// epilogue, GEMM-2 with fp32 y) as tcgen05 MMAs of M = 256 spread over the
// two SMs of a TPC (.cta_group::2). This is the "分组 GMM" / FusedMoEGMM step
// of "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5 (the
// routed path is the bulk of the MoE block's time), for groups with many
// rows.
//
//   GEMM-1 (MODE 0):  h[r, i] = silu(sum_c a[r,c] Wg[g,i,c]) * (sum_c a[r,c] Wu[g,i,c])
//   GEMM-2 (MODE 1):  y[r, m] = sum_i h[r,i] Wd[g,m,i]
//
// Why pairs: with one SM per MMA, a 128 x 256 tile needs 48 KB of operands
// per 64-wide K slice, and the ring of stages that fits in shared memory
// cannot hold enough of them in flight to keep the tensor pipe busy. In a
// pair each SM stages its own half of both operands and the MMA reads the
// other half from the peer SM, so a K slice costs each SM less shared memory
// for the same tensor work.
//
// Tiling (weights as M): the pair's 256 MMA rows are weight rows and N is a
// chunk of the group's rows (tokens), up to 256, cut to the chunk rounded up
// to 32 so a group's last chunk wastes little. GEMM-1: each SM's 128 rows
// hold the gate and up rows of 64 intermediate features, interleaved by 16 so
// that every 32-row quarter (the TMEM lanes one epilogue warp reads) has the
// gate rows of 16 features followed by their up rows; one accumulator then
// holds both halves of SwiGLU and a lane finds its partner by a shuffle (a
// pair tile covers 128 features). GEMM-2: 128 rows of W_down per SM (256
// hidden features per pair tile). Each SM stages N/2 token rows; in each SM's TMEM, lane = weight
// row, column = token (columns 0..N/2-1 from the even CTA's rows, N/2..N-1
// from the odd's). One MMA per 16-wide K step keeps the single issuing thread
// ahead of the tensor pipe.
//
// Roles in each CTA (192 threads): warp 0 lane 0 of each CTA loads its
// halves by TMA into local stages (local full barriers); warp 1 lane 0 of the
// odd CTA relays each landed stage to the leader's full barrier for that
// stage, which therefore completes once both halves are in; warp 1 lane 0 of
// the even CTA (leader) waits on it, issues the pair MMAs and commits to both
// CTAs' empty and accumulator barriers; warps 2-5 of both CTAs read their TMEM lanes and store h / y,
// then tell the leader the accumulator is free. All waits are bounded (about
// 2 s): on expiry the CTA records an error code, raises its abort flag,
// drains its in-flight copies (the leader its MMAs), and both CTAs meet at a
// cluster barrier before freeing TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "internal.h"
#include "gemm_sched.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;           // K elements per sub-tile: one 128-byte swizzle row of bf16
constexpr int kKSub = 2;          // sub-tiles per stage: 128 K elements per stage
constexpr int kMaxGroups = 1024;
constexpr int kMaxSmem = 232448;  // 227 KB dynamic shared memory per CTA
constexpr uint16_t kPairMask = 0x3;

template <int MODE>
struct PairGeo {
  static constexpr int W_ROWS = 128;                  // weight rows per CTA (half of M = 256)
  static constexpr int F_CTA = MODE == 0 ? 64 : 128;  // output features per CTA
  static constexpr int W_COLS = 2 * F_CTA;            // output features per pair tile
  static constexpr int NT = 256;                      // tokens per pair tile at most (N)
  static constexpr int B_ROWS = NT / 2;               // token rows each CTA stages
  static constexpr int A_BYTES = W_ROWS * 128;        // 16 KB: one A sub-tile
  static constexpr int B_BYTES = B_ROWS * 128;        // 16 KB: one B sub-tile
  static constexpr int STAGE_BYTES = kKSub * (A_BYTES + B_BYTES);
  static constexpr int ACC_COLS = NT;                 // TMEM columns per accumulator buffer
  static constexpr int W_BOX = MODE == 0 ? 16 : 128;  // rows per weight TMA box
  static constexpr int TMEM_COLS = 512;
  // GEMM-1 stages 16 weight boxes per stage; a second producer warp (warp 6)
  // issues the up boxes so that TMA issue keeps pace with the MMAs.
  static constexpr int THREADS = MODE == 0 ? 224 : 192;
  static constexpr int TABLE_BYTES = 2 * (kMaxGroups + 8) * 4;  // tile starts, row starts
  static constexpr int BAR_BYTES = 512;
  // Shared memory: the A tiles of every stage, then the B tiles of every
  // stage, then the tile table and barriers, then SLACK unused bytes. Each
  // MMA reads its CTA's half of A and of B; with this order even a read of
  // twice those halves would stay inside the allocation.
  static constexpr int SLACK = 16384;
  static constexpr int EXTRA = 1024 + TABLE_BYTES + BAR_BYTES + SLACK;
  static constexpr int S_FREE = (kMaxSmem - EXTRA) / STAGE_BYTES;
  static constexpr int S = S_FREE > 8 ? 8 : S_FREE;
  static constexpr int A_REGION = S * kKSub * A_BYTES;
  static constexpr int RING_BYTES = S * STAGE_BYTES;
  static constexpr int SMEM = EXTRA + RING_BYTES;
  static_assert(SLACK >= B_BYTES && SLACK >= A_BYTES, "slack covers a doubled read");
  static constexpr int NBARS = 2 * S + 5;  // full, empty [S]; tfull[2], tempty[2], drain
  static_assert(S >= 3, "ring too shallow");
  static_assert(A_REGION + S * kKSub * B_BYTES == RING_BYTES, "ring layout");
  static_assert(2 * ACC_COLS <= TMEM_COLS, "two accumulator buffers");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1024-byte alignment of swizzled tiles");
  static_assert(NBARS * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(SMEM <= kMaxSmem, "shared memory budget");
};

// Tokens of the tile's chunk and the MMA's N. A group of r rows is cut into
// ceil(r / NT) chunks of one size (r / chunks rounded up to 32, so each CTA's
// half is a multiple of 16 rows), the last taking the rest: 341 rows give
// 192 + 149 rather than 256 + 85, so neither chunk leaves the tensor pipe
// waiting on the issuing thread. N is the chunk rounded up to 32.
template <int NT>
__device__ __forceinline__ void chunk_of(const TileInfo& ti, int& tok0, int& ntok, int& n) {
  const int chunks = (ti.nrows + NT - 1) / NT;
  const int cs = ((ti.nrows + chunks - 1) / chunks + 31) & ~31;
  tok0 = ti.tt * cs;
  const int left = ti.nrows - tok0;
  ntok = left < cs ? left : cs;
  n = (ntok + 31) & ~31;
}

// One tile's epilogue, executed by one warp for its 32 TMEM lanes.
// GEMM-1: lanes 0-15 hold the gate rows and lanes 16-31 the up rows of the
// warp's 16 features. Lane l and lane l ^ 16 swap values by a shuffle so that
// each has (gate, up) for one feature at 16 of every 32 tokens (lanes 0-15
// the first 16, lanes 16-31 the last 16), and each stores silu(g) * u.
// GEMM-2: every lane stores its row of W_down's output as y.
template <int MODE>
__device__ __forceinline__ void epilogue_pair(const KParams& p, const TileInfo& ti, uint32_t tb,
                                              int q, int lane, uint32_t rank) {
  using Gm = PairGeo<MODE>;
  int tok0, ntok, n;
  chunk_of<Gm::NT>(ti, tok0, ntok, n);
  const size_t row0 = (size_t)ti.row0 + tok0;
  if (MODE == 0) {
    const bool up_lane = lane >= 16;
    const int f = ti.wt * Gm::W_COLS + (int)rank * Gm::F_CTA + q * 16 + (lane & 15);
    const bool fv = f < p.N;
    const int jbase = up_lane ? 16 : 0;
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
    for (int c = 0; c < n; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tb + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        // A gate lane keeps token j and sends token j + 16; an up lane keeps
        // token j + 16 and sends token j.
        const float keep = __uint_as_float(up_lane ? v[j + 16] : v[j]);
        const float send = __uint_as_float(up_lane ? v[j] : v[j + 16]);
        const float other = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
        const float g = up_lane ? other : keep;
        const float u = up_lane ? keep : other;
        const int r = c + jbase + j;
        if (r < ntok && fv) h[(row0 + r) * p.N + f] = __float2bfloat16_rn(silu_f(g) * u);
      }
    }
  } else {
    const int f = ti.wt * Gm::W_COLS + (int)rank * Gm::F_CTA + q * 32 + lane;
    const bool fv = f < p.N;
    float* y = static_cast<float*>(p.out);
#pragma unroll 1
    for (int c = 0; c < n; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tb + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int r = c + j;
        if (r < ntok && fv) y[(row0 + r) * p.N + f] = __uint_as_float(v[j]);
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(PairGeo<MODE>::THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_act,
                             const __grid_constant__ CUtensorMap map_w0,
                             const __grid_constant__ CUtensorMap map_w1, const KParams p) {
  using Gm = PairGeo<MODE>;
  constexpr int NS = Gm::S;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* base = smem_raw + pad;
  const uint32_t base_u32 = raw_addr + pad;
  // Shared memory: A tiles | B tiles | tile table | barriers, TMEM address,
  // abort flag | slack. The layout is the same in both CTAs, so a
  // descriptor's offsets address the matching half in the peer.
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + Gm::RING_BYTES);
  int32_t* row_start = tile_start + kMaxGroups + 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Gm::RING_BYTES + Gm::TABLE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Gm::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // full[s]: in the leader two arrivals (its producer's, with the stage's
  // bytes, and the peer's relay once the peer's half has landed); in the
  // peer one (its producer's).
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NS + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NS + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NS + 2 + a); };  // leader: 8 epilogue warps
  const uint32_t drain_bar = bar0 + 8u * (2 * NS + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: leader, 1: peer
  const int pair = (int)cluster_id_x(), npairs = (int)ncluster_x();

  // ---- tile table: tile_start[g] = tiles of groups before g.
  const int n_wt = (p.N + Gm::W_COLS - 1) / Gm::W_COLS;
  for (int g = threadIdx.x; g < p.G; g += Gm::THREADS) {
    int r0, nr;
    group_rows(p, g, r0, nr);
    tile_start[g] = n_wt * ((nr + Gm::NT - 1) / Gm::NT);
  }
  fill_row_start(p, row_start, threadIdx.x, Gm::THREADS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full_bar(s), rank == 0 ? 2 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // one warp of each CTA of the pair, together
    tmem_alloc_pair(smem_u32(tmem_slot), Gm::TMEM_COLS);
    tmem_relinquish_pair();
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
  // Both CTAs' barriers are initialised and the pair's TMEM is allocated
  // before either CTA signals the other.
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[p.G];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring rg;
      Armed armed;
      bool ok = true;
      const int n_stages = (p.num_kb + kKSub - 1) / kKSub;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const TileInfo ti = decode_tile_s<Gm::NT>(p.G, tile_start, row_start, tile);
        int tok0, ntok, n;
        chunk_of<Gm::NT>(ti, tok0, ntok, n);
        const int act_row = ti.row0 + tok0 + (int)rank * (n / 2);
        // First weight row of this CTA's A tile: GEMM-1 the gate and up rows of
        // 64 features, GEMM-2 128 rows of W_down.
        const int w_row = ti.g * p.N + ti.wt * Gm::W_COLS + (int)rank * Gm::F_CTA;
        for (int kb = 0; kb < n_stages; ++kb) {
          if (!mbar_wait_bounded_cluster(empty_bar(rg.s), rg.ph ^ 1u, abort_flag, p.status,
                                         MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const int nsub = p.num_kb - kb * kKSub < kKSub ? p.num_kb - kb * kKSub : kKSub;
          const uint32_t fb = full_bar(rg.s);
          mbar_arrive_expect_tx(fb, (uint32_t)nsub * (Gm::A_BYTES + Gm::B_BYTES));
          for (int j = 0; j < nsub; ++j) {
            const int kx = (kb * kKSub + j) * kBK;
            const uint32_t sA = base_u32 + (rg.s * kKSub + j) * Gm::A_BYTES;
            if (MODE == 0) {
              // Quarter t of the A sub-tile (32 rows, 4 KB): gate rows of
              // features 16t .. 16t+15, then their up rows (warp 6 loads those).
#pragma unroll
              for (int t = 0; t < 4; ++t) tma_load_2d(sA + t * 4096, &map_w0, fb, kx, w_row + 16 * t);
            } else {
              tma_load_2d(sA, &map_w0, fb, kx, w_row);
            }
            tma_load_2d(base_u32 + Gm::A_REGION + (rg.s * kKSub + j) * Gm::B_BYTES, &map_act, fb, kx,
                        act_row);
          }
          armed.mark(rg);
          rg.next(NS);
        }
      }
      if (!ok) {  // let copies already issued land before the CTA leaves
        for (int s = 0; s < NS; ++s)
          if (armed.mask & (1u << s)) drain_wait(full_bar(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp walks the loop in step, so tile, stage and descriptor
      // values are warp-uniform; lane 0 polls the barriers (the result is
      // broadcast) and issues the tcgen05 instructions.
      auto wait_all = [&](uint32_t bar, uint32_t parity) {
        int v = 0;
        if (lane == 0)
          v = mbar_wait_bounded_cluster(bar, parity, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA,
                                        p.limit_ns) ? 1 : 0;
        return __shfl_sync(0xFFFFFFFFu, v, 0) != 0;
      };
      Ring rg;
      bool ok = true, issued = false;
      int local = 0;
      const int n_stages = (p.num_kb + kKSub - 1) / kKSub;
      for (int tile = pair; ok && tile < total; tile += npairs, ++local) {
        const TileInfo ti = decode_tile_s<Gm::NT>(p.G, tile_start, row_start, tile);
        int tok0, ntok, n;
        chunk_of<Gm::NT>(ti, tok0, ntok, n);
        const uint32_t idesc = idesc_bf16_f32(256, n);
        const int acc = local & 1;
        const uint32_t ap = (uint32_t)(local >> 1) & 1u;
        if (!wait_all(tempty_bar(acc), ap ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * Gm::ACC_COLS);
        for (int kb = 0; kb < n_stages; ++kb) {
          // Both halves of the stage: the leader's bytes and the peer's relay.
          if (!wait_all(full_bar(rg.s), rg.ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = p.num_kb - kb * kKSub < kKSub ? p.num_kb - kb * kKSub : kKSub;
          // Descriptors of the stage's first 16-wide K step; each further step
          // is 32 bytes on (+2 in the start-address field), the second
          // sub-tile 16 KB on (+1024).
          const uint64_t a0 = sw128_kmajor_desc(base_u32 + rg.s * kKSub * Gm::A_BYTES);
          const uint64_t b0 = sw128_kmajor_desc(base_u32 + Gm::A_REGION + rg.s * kKSub * Gm::B_BYTES);
          if (lane == 0) {
            for (int j = 0; j < nsub; ++j) {
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                umma_bf16_pair(d, a0 + (uint64_t)(j * (Gm::A_BYTES >> 4) + 2 * k),
                               b0 + (uint64_t)(j * (Gm::B_BYTES >> 4) + 2 * k), idesc,
                               (kb | j | k) ? 1u : 0u);
            }
            umma_commit_pair_mc(empty_bar(rg.s), kPairMask);
          }
          __syncwarp();
          issued = true;
          rg.next(NS);
        }
        if (!ok) break;
        if (lane == 0) umma_commit_pair_mc(tfull_bar(acc), kPairMask);
        __syncwarp();
      }
      // Every MMA reads both CTAs' shared memory and writes both TMEMs: all
      // of them complete before either CTA goes on to leave.
      if (issued && lane == 0) {
        umma_commit_pair(drain_bar);
        drain_wait(drain_bar, 0, 200000000ull);
      }
    } else if (lane == 0) {
      // ---------------------------------------------------------- relay (peer)
      // Report each landed stage of this CTA's half to the leader's MMA thread.
      Ring rg;
      bool ok = true;
      const int n_stages = (p.num_kb + kKSub - 1) / kKSub;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        for (int kb = 0; kb < n_stages; ++kb) {
          if (!mbar_wait_bounded(full_bar(rg.s), rg.ph, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA,
                                 p.limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_remote(mapa_shared(full_bar(rg.s), 0));
          rg.next(NS);
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ up boxes (GEMM-1)
    if (MODE == 0 && lane == 0) {
      Ring rg;
      Armed armed;
      bool ok = true;
      const int n_stages = (p.num_kb + kKSub - 1) / kKSub;
      for (int tile = pair; ok && tile < total; tile += npairs) {
        const TileInfo ti = decode_tile_s<Gm::NT>(p.G, tile_start, row_start, tile);
        const int w_row = ti.g * p.N + ti.wt * Gm::W_COLS + (int)rank * Gm::F_CTA;
        for (int kb = 0; kb < n_stages; ++kb) {
          if (!mbar_wait_bounded_cluster(empty_bar(rg.s), rg.ph ^ 1u, abort_flag, p.status,
                                         MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const int nsub = p.num_kb - kb * kKSub < kKSub ? p.num_kb - kb * kKSub : kKSub;
          const uint32_t fb = full_bar(rg.s);  // bytes counted by warp 0's expect_tx
          for (int j = 0; j < nsub; ++j) {
            const int kx = (kb * kKSub + j) * kBK;
            const uint32_t sA = base_u32 + (rg.s * kKSub + j) * Gm::A_BYTES;
#pragma unroll
            for (int t = 0; t < 4; ++t)
              tma_load_2d(sA + t * 4096 + 2048, &map_w1, fb, kx, w_row + 16 * t);
          }
          armed.mark(rg);
          rg.next(NS);
        }
      }
      if (!ok) {
        for (int s = 0; s < NS; ++s)
          if (armed.mask & (1u << s)) drain_wait(full_bar(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
    int local = 0;
    for (int tile = pair; tile < total; tile += npairs, ++local) {
      const int acc = local & 1;
      const uint32_t ap = (uint32_t)(local >> 1) & 1u;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded_cluster(tfull_bar(acc), ap, abort_flag, p.status,
                                       MOE_DEV_TIMEOUT_EPILOGUE, p.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = decode_tile_s<Gm::NT>(p.G, tile_start, row_start, tile);
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * Gm::ACC_COLS);
      epilogue_pair<MODE>(p, ti, tb, q, lane, rank);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
      }
    }
  }

  // Both CTAs arrive here only after their roles are done (every wait above
  // is bounded), so neither frees TMEM or leaves while the other may still
  // touch its shared memory or barriers.
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Gm::TMEM_COLS);
  }
}

}  // namespace

template <int MODE>
static cudaError_t run_gemm_pair(const GroupedGemmArgs& a, cudaStream_t s) {
  using Gm = PairGeo<MODE>;
  const int Kdim = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const void* act = MODE == 0 ? a.a : a.h;
  const void* w0 = MODE == 0 ? a.w_gate : a.w_down;
  const void* w1 = MODE == 0 ? a.w_up : a.w_down;
  if (a.rows == 0 || a.G == 0) return cudaSuccess;
  const int G = a.offsets ? a.G : 1;
  CUtensorMap m_act, m_w0, m_w1;
  if (!make_tmap_bf16(&m_act, act, Kdim, a.rows, Gm::B_ROWS) ||
      !make_tmap_bf16(&m_w0, w0, Kdim, (uint64_t)G * N, Gm::W_BOX) ||
      !make_tmap_bf16(&m_w1, w1, Kdim, (uint64_t)G * N, Gm::W_BOX))
    return cudaErrorInvalidValue;
  KParams p = {};
  p.offsets = a.offsets;
  p.G = G;
  p.rows = a.rows;
  p.num_kb = (Kdim + kBK - 1) / kBK;
  p.N = N;
  p.out = MODE == 0 ? a.h : static_cast<void*>(a.y);
  p.status = a.status;
  p.limit_ns = a.wait_limit_ns;
  p.fold_group = -1;
  const long long n_wt = (N + Gm::W_COLS - 1) / Gm::W_COLS;
  const long long max_tiles = n_wt * ((a.rows + Gm::NT - 1) / Gm::NT + G);
  const long long pairs_cap = a.num_sms / 2;
  const int pairs = (int)(max_tiles < pairs_cap ? max_tiles : pairs_cap);
  if (pairs < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(Gm::THREADS, 1, 1);
  cfg.dynamicSmemBytes = Gm::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE>, m_act, m_w0, m_w1, p);
}

bool gemm_pair_supported(const GroupedGemmArgs& a) {
  // Bases of the operand tensor maps are 16-byte aligned (checked by the API)
  // and the K extents are multiples of 64 (H, I % 64 == 0).
  return a.num_sms >= 2 && a.shared_w_gate == nullptr;
}

cudaError_t gemm_pair_prepare_device() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<0>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, PairGeo<0>::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairGeo<1>::SMEM);
  return e;
}

cudaError_t launch_gemm_pair_gate_up(const GroupedGemmArgs& a, cudaStream_t s) {
  return run_gemm_pair<0>(a, s);
}

cudaError_t launch_gemm_pair_down(const GroupedGemmArgs& a, cudaStream_t s) {
  return run_gemm_pair<1>(a, s);
}

}  // namespace moe
