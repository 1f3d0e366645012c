// Step 3's GEMMs in MX formats with a wide weight tile: the same products as
// grouped_gemm_mx_kernel<MODE, W4> (gemm_mx.cu; "腾讯混元 Hy3 在 CANN NPU 上的
// 高性能推理部署与优化实战", section 8.2: W8A8 MXFP8 and the W4A8 recipe with
// MXFP4 routed weights), but each MMA covers N = 256 weight rows instead of 128:
//   MODE 0 (GEMM-1): gate 128 + up 128 rows, h = silu(x Wg^T) * (x Wu^T) for
//                    128 columns of h, re-quantised to MXFP8 per 32 along I;
//   MODE 1 (GEMM-2): 256 rows of W_down, y = h Wd^T for 256 columns, fp32,
//                    staged per warp through shared memory and stored as
//                    64-byte row segments.
//
// What sets the pace of these kernels is how much each issuing thread does
// per K stage: every tcgen05 instruction, barrier wait and TMA issue costs
// its thread tens to a couple of hundred cycles (clock64 traces of each role),
// and a stage carries 536 cycles of tensor work at N = 256 (268 at N = 128).
// At N = 128 the MMA thread alone (4 MMAs, a commit, the waits) needed ~620
// cycles per stage. So this kernel doubles the work per MMA and keeps every
// role's per-stage work short:
//   - the MMA thread waits on one barrier per stage (weights, activations and
//     the stage's scales in TMEM), issues 4 MMAs from precomputed descriptors
//     and one commit, which frees the weight stage, the activation stage and
//     the TMEM scale slot at once (their rings are tied to the weight ring);
//   - with E2M1 weights in tile order (moe_tile_mxfp4_weights) a stage's 256
//     weight rows are one contiguous 16 KB block and one TMA load;
//   - scale atoms are fetched two stages per bulk copy, two groups ahead of
//     their data, and a scale warp moves them into TMEM slots ahead of the MMA
//     (a tcgen05.cp waits in the tensor pipe behind the MMAs issued before it,
//     so one issued after the previous stage's MMAs would stall the next).
//
// TMEM: one 256-column fp32 accumulator plus the scale slots, so the
// accumulator is single-buffered. Eight epilogue warps (two per TMEM lane
// quarter) copy it into registers at once (128 values a thread), hand it back
// to the MMA thread, and only then compute SwiGLU and the MXFP8 codes.
//
// Weight-row order inside a tile follows the packed scale atoms of GEMM-1
// (gate and up interleaved per 64 rows, mx_layout.cuh / moe_pack_mx_scales):
// B rows 0-63 gate, 64-127 up (atom 2 wt), 128-191 gate, 192-255 up (atom
// 2 wt + 1), so the two B atoms of a K block land in TMEM scale columns 0-3
// and 4-7 unchanged (the scale of B column n in column n / 32, lane n % 32).
//
// Persistent, one CTA per SM, 384 threads:
//   warp 0      weight producer: per 128-wide K stage the stage's weight rows
//               (one box for E2M1 in tile order, four for row-major E4M3),
//               4-stage ring; and the scale atoms of stage pairs two groups
//               ahead.
//   warp 11     activation producer: the A tile (128 token rows), completing
//               on the weight stage's barrier (4-stage ring; mostly L2 hits: a
//               token tile is read by every weight tile of its expert).
//   warp 2      scale warp: three tcgen05.cp per stage into the stage's slot.
//   warp 1      TMEM allocator + MMA issuer: 4 MMAs (K = 32) per stage.
//   warps 3-10  epilogue: warp w reads TMEM lane quarter w % 4 and accumulator
//               columns 128 * ((w - 3) / 4) .. +127: GEMM-1 h columns 64 of
//               them, GEMM-2 128 y columns (through a 2 KB staging block).
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

constexpr int wStagesB = 4;               // weight ring; also the TMEM scale slots
constexpr int wStagesA = 4;               // activation ring (one slot per weight slot: measured
                                          // faster than 5 + 3, the activation loads wait on L2 too)
constexpr int wGroup = 2;                 // K stages per atom group (one bulk copy per atom kind)
constexpr int wGroupSlots = 4;            // atom groups in shared memory
constexpr int wGroupAhead = 2;            // groups between an atom group's load and its first stage
constexpr int wThreads = 384;
constexpr int wScaleWarp = 2;
constexpr int wEpiWarp0 = 3;
constexpr int wEpiWarps = 8;
constexpr int wProdAWarp = 11;
constexpr int wATile = 128 * 128;         // 128 token rows x 128 K bytes
constexpr int wBTile = 256 * 128;         // 256 weight rows x 128 K slots
constexpr int wBox = 64 * 128;            // one 64-row E4M3 weight box in shared memory
constexpr int wGroupBytes = 3 * wGroup * kAtomBytes;  // A atoms | B atoms (rows 0-127) | B atoms (128-255)
constexpr int wAccCols = 256;
constexpr int wSfCol0 = wAccCols;         // TMEM scale slot s: wSfCol0 + 16 s (A +0..3, B +8..15)
constexpr int wTmemCols = 512;
constexpr int wMaxGroups = 512;
constexpr int wTableBytes = 2 * (wMaxGroups + 8) * 4;  // tile starts + group row starts
constexpr int wNumBars = 2 * wStagesB + 2 * wGroupSlots + 4;
constexpr int wBarBytes = 256;
// Shared memory: weight ring | activation ring | atom groups | tables | barriers.
constexpr int wOffA = wStagesB * wBTile;
constexpr int wOffSf = wOffA + wStagesA * wATile;
constexpr int wOffTable = wOffSf + wGroupSlots * wGroupBytes;
constexpr int wOffBars = wOffTable + wTableBytes;
// GEMM-2 epilogue staging after the barriers: one 32-row x 16-column fp32 block
// (2 KB) per epilogue warp.
constexpr int wStgWarp = 32 * 16;          // floats
constexpr int wOffStg = wOffBars + wBarBytes;
template <int MODE>
constexpr int wSmemFor() { return 1024 + wOffStg + (MODE == 1 ? wEpiWarps * wStgWarp * 4 : 0); }
constexpr int wSmem = wSmemFor<0>();
static_assert(wSmemFor<1>() <= 232448, "shared memory budget");
static_assert(wOffStg % 16 == 0, "16-byte staging stores");
static_assert(wSfCol0 + 16 * wStagesB <= wTmemCols, "TMEM budget");
static_assert(wNumBars * 8 + 8 <= wBarBytes, "barrier area");
static_assert(wStagesA <= wStagesB, "an activation slot is freed by a weight-ring phase no later than its own");
static_assert(wGroupAhead < wGroupSlots, "an atom group slot is reloaded only after its copies");
static_assert(wThreads == 32 * (wProdAWarp + 1) && wEpiWarp0 + wEpiWarps == wProdAWarp, "warp roles");

// h = silu(g) * u for one 32-column block of a row, as MXFP8 codes + E8M0.
__device__ __forceinline__ void store_h_block(const uint32_t (&g)[32], const uint32_t (&u)[32],
                                              uint8_t* dst, uint8_t* scale_dst) {
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
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  *scale_dst = (uint8_t)code;
}

// Parity of the phase of a ring barrier that completes for the n-th time
// (n = 0, 1, ...) when stage n * depth + slot completes.
__device__ __forceinline__ uint32_t round_parity(int stage, int depth) { return (uint32_t)(stage / depth) & 1u; }

template <int MODE, bool W4>
__global__ void __launch_bounds__(wThreads, 1)
    grouped_gemm_mx_wide_kernel(const __grid_constant__ CUtensorMap map_act,
                                const __grid_constant__ CUtensorMap map_w0,
                                const __grid_constant__ CUtensorMap map_w1, const KParams p) {
  // Transaction bytes of a stage on its weight barrier: the weights (E2M1
  // boxes count their packed global bytes, half their shared-memory
  // footprint) and the activation tile.
  constexpr uint32_t kTxStage = (W4 ? wBTile / 2 : wBTile) + wATile;
  constexpr uint32_t kIdescFmt = W4 ? (5u << 10) : 0u;  // B format: E2M1 or E4M3
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = ((raw_addr + 1023u) & ~1023u) - raw_addr;
  uint8_t* base = smem_raw + pad;
  const uint32_t sm0 = raw_addr + pad;
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + wOffTable);
  int32_t* row_start = tile_start + (wMaxGroups + 8);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + wOffBars);
  float* y_stage = reinterpret_cast<float*>(base + wOffStg);  // GEMM-2 only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + wNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // full(s): stage s's weights and activations landed and its scales are in
  // TMEM slot s (two arrivals: the weight producer's, with both producers'
  // bytes, and the scale warp's commit); empty(s): its MMAs are done (frees
  // the weight stage, the activation stage of the same K stage and TMEM scale
  // slot s).
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (wStagesB + s); };
  // gfull(g): atom group slot g landed; gfree(g): its copies into TMEM are done.
  auto gfull = [&](int g) { return bar0 + 8u * (2 * wStagesB + g); };
  auto gfree = [&](int g) { return bar0 + 8u * (2 * wStagesB + wGroupSlots + g); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * wStagesB + 2 * wGroupSlots);
  const uint32_t tempty_bar = tfull_bar + 8u;
  const uint32_t drain_bar = tfull_bar + 16u;
  const uint32_t sdrain_bar = tfull_bar + 24u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Output columns per tile: GEMM-1 128 of h (N = I % 128 == 0), GEMM-2 256 of y (N = H % 256 == 0).
  constexpr int kCols = MODE == 0 ? 128 : 256;
  const int n_wt = p.N / kCols;
  fill_row_start(p, row_start, threadIdx.x, wThreads);
  for (int g = threadIdx.x; g < p.G; g += wThreads) {
    int r0, nr;
    group_rows(p, g, r0, nr);
    tile_start[g] = n_wt * ((nr + 127) / 128);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < wStagesB; ++s) {
      mbar_init(full(s), 2);  // the weight producer's arrival (both producers' bytes) + the scale commit
      mbar_init(empty(s), 1);
    }
    for (int g = 0; g < wGroupSlots; ++g) {
      mbar_init(gfull(g), 1);
      mbar_init(gfree(g), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, wEpiWarps);
    mbar_init(drain_bar, 1);
    mbar_init(sdrain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), wTmemCols);
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
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      Armed armed, armed_g;
      bool ok = true;
      // Atom groups: a group is up to wGroup consecutive K stages of one tile.
      int g_tile = blockIdx.x, g_kb = 0, nload = 0;
      TileInfo g_ti{};
      if (g_tile < total) g_ti = decode_tile_s<128>(p.G, tile_start, row_start, g_tile);
      auto load_group = [&]() -> bool {
        if (g_tile >= total) return true;
        const int gs = nload % wGroupSlots;
        if (nload >= wGroupSlots &&
            !mbar_wait_bounded(gfree(gs), round_parity(nload - wGroupSlots, wGroupSlots), abort_flag, p.status,
                               MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns))
          return false;
        const int cnt = n_k - g_kb < wGroup ? n_k - g_kb : wGroup;
        const uint32_t bytes = (uint32_t)cnt * kAtomBytes;
        const long long a_blk = tile_start[g_ti.g] / n_wt + g_ti.tt;
        // Weight atoms b_blk, b_blk + 1: GEMM-1 the gate/up atom matrix (2N rows per
        // group), GEMM-2 the down atoms (N rows per group).
        const long long b_blk = (long long)g_ti.g * ((MODE == 0 ? 2 : 1) * p.N / 128) + 2 * g_ti.wt;
        const uint8_t* a_atom = p.s_act + (a_blk * n_k + g_kb) * kAtomBytes;
        const uint8_t* b_atom = p.s_w0 + (b_blk * n_k + g_kb) * kAtomBytes;
        const uint32_t dst = sm0 + wOffSf + gs * wGroupBytes;
        const uint32_t fb = gfull(gs);
        mbar_arrive_expect_tx(fb, 3 * bytes);
        bulk_load_hint(dst, a_atom, bytes, fb, pol);
        bulk_load_hint(dst + wGroup * kAtomBytes, b_atom, bytes, fb, pol);
        bulk_load_hint(dst + 2 * wGroup * kAtomBytes, b_atom + (size_t)n_k * kAtomBytes, bytes, fb, pol);
        Ring at;
        at.s = gs;
        at.ph = round_parity(nload, wGroupSlots);
        armed_g.mark(at);
        ++nload;
        g_kb += cnt;
        if (g_kb == n_k) {
          g_kb = 0;
          g_tile += gridDim.x;
          if (g_tile < total) g_ti = decode_tile_s<128>(p.G, tile_start, row_start, g_tile);
        }
        return true;
      };
      for (int i = 0; ok && i < wGroupAhead; ++i) ok = load_group();
      int j = 0;  // stage
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile_s<128>(p.G, tile_start, row_start, tile);
        const int w_row = ti.g * p.N + ti.wt * kCols;
        // Tile order: GEMM-1 the gate/up pair block t (256 rows), GEMM-2 the
        // 128-row down blocks t and t + 1.
        const int t = MODE == 0 ? ti.g * n_wt + ti.wt : (ti.g * p.N + ti.wt * kCols) / 128;
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          if (kb % wGroup == 0 && !load_group()) {
            ok = false;
            break;
          }
          const int s = j % wStagesB;
          if (j >= wStagesB && !mbar_wait_bounded(empty(s), round_parity(j - wStagesB, wStagesB), abort_flag,
                                                  p.status, MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full(s);
          mbar_arrive_expect_tx(fb, kTxStage);
          const uint32_t st = sm0 + s * wBTile;
          if (W4) {
            if (MODE == 0) {
              tma_load_2d_hint(st, &map_w0, fb, 0, (t * n_k + kb) * 256, pol);
            } else {
              tma_load_2d_hint(st, &map_w0, fb, 0, (t * n_k + kb) * 128, pol);
              tma_load_2d_hint(st + 2 * wBox, &map_w0, fb, 0, ((t + 1) * n_k + kb) * 128, pol);
            }
          } else {
            // Row-major E4M3, four 64-row boxes: GEMM-1 gate, up, gate, up (64 rows
            // each, the atoms' order); GEMM-2 256 consecutive down rows.
            const int kx = kb * 128;
            const CUtensorMap* m1 = MODE == 0 ? &map_w1 : &map_w0;
            const int r1 = MODE == 0 ? 0 : 64;
            tma_load_2d_hint(st, &map_w0, fb, kx, w_row, pol);
            tma_load_2d_hint(st + wBox, m1, fb, kx, w_row + r1, pol);
            tma_load_2d_hint(st + 2 * wBox, &map_w0, fb, kx, w_row + (MODE == 0 ? 64 : 128), pol);
            tma_load_2d_hint(st + 3 * wBox, m1, fb, kx, w_row + (MODE == 0 ? 64 : 192), pol);
          }
          Ring r;
          r.s = s;
          r.ph = round_parity(j, wStagesB);
          armed.mark(r);
        }
      }
      if (!ok) {
        for (int s = 0; s < wStagesB; ++s)
          if (armed.mask & (1u << s)) drain_wait(full(s), (armed.phase >> s) & 1u, 100000000ull);
        for (int g = 0; g < wGroupSlots; ++g)
          if (armed_g.mask & (1u << g)) drain_wait(gfull(g), (armed_g.phase >> g) & 1u, 100000000ull);
      }
    }
  } else if (warp == wProdAWarp) {
    // ------------------------------------------------------------ activation producer
    if (lane == 0) {
      bool ok = true;
      Armed armed;
      int j = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile_s<128>(p.G, tile_start, row_start, tile);
        const int act_row = ti.row0 + ti.tt * 128;
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          // Activation slot j % wStagesA last held stage j - wStagesA; its MMAs
          // completed the weight ring's empty barrier of that stage. Those MMAs
          // also imply stage j - wStagesB's, so the phase of full(j % wStagesB)
          // this load completes on is already the current one.
          if (j >= wStagesA) {
            const int prev = j - wStagesA;
            if (!mbar_wait_bounded(empty(prev % wStagesB), round_parity(prev, wStagesB), abort_flag, p.status,
                                   MOE_DEV_TIMEOUT_PRODUCER, p.limit_ns)) {
              ok = false;
              break;
            }
          }
          tma_load_2d(sm0 + wOffA + (j % wStagesA) * wATile, &map_act, full(j % wStagesB), kb * 128, act_row);
          Ring r;
          r.s = j % wStagesB;
          r.ph = round_parity(j, wStagesB);
          armed.mark(r);
        }
      }
      if (!ok) {  // bounded: a stage the weight producer never armed does not complete
        for (int s = 0; s < wStagesB; ++s)
          if (armed.mask & (1u << s)) drain_wait(full(s), (armed.phase >> s) & 1u, 100000000ull);
      }
    }
  } else if (warp == wScaleWarp) {
    // ------------------------------------------------------------ scale warp
    if (lane == 0) {
      bool ok = true, issued = false;
      int j = 0, ng = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          const int gs = ng % wGroupSlots;
          const int i = kb % wGroup;  // stage within its atom group
          const bool last = i == wGroup - 1 || kb == n_k - 1;
          const int s = j % wStagesB;
          // The group's atoms have landed; TMEM slot s is free once the MMAs
          // of stage j - wStagesB are done.
          if ((i == 0 && !mbar_wait_bounded(gfull(gs), round_parity(ng, wGroupSlots), abort_flag, p.status,
                                            MOE_DEV_TIMEOUT_MMA, p.limit_ns)) ||
              (j >= wStagesB && !mbar_wait_bounded(empty(s), round_parity(j - wStagesB, wStagesB), abort_flag,
                                                   p.status, MOE_DEV_TIMEOUT_MMA, p.limit_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tmem_base + (uint32_t)(wSfCol0 + 16 * s);
          const uint32_t src = sm0 + wOffSf + gs * wGroupBytes + i * kAtomBytes;
          tmem_cp_32x128b_warpx4(sf, src);
          tmem_cp_32x128b_warpx4(sf + 8, src + wGroup * kAtomBytes);
          tmem_cp_32x128b_warpx4(sf + 12, src + 2 * wGroup * kAtomBytes);
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true, issued = false;
      int local = 0, j = 0;
      constexpr uint32_t kIdesc0 = idesc_mxf8_e4m3(128, 256, 0, 0) | kIdescFmt;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        // The single accumulator is free once the epilogue copied the last tile out.
        if (!mbar_wait_bounded(tempty_bar, ((uint32_t)local & 1u) ^ 1u, abort_flag, p.status,
                               MOE_DEV_TIMEOUT_MMA, p.limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < n_k; ++kb, ++j) {
          const int s = j % wStagesB;
          const uint32_t ph = round_parity(j, wStagesB);
          if (!mbar_wait_bounded(full(s), ph, abort_flag, p.status, MOE_DEV_TIMEOUT_MMA, p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Descriptors of the stage's operands; +32 bytes along K is +2 in
          // the start-address field.
          const uint64_t da = sw128_kmajor_desc(sm0 + wOffA + (j % wStagesA) * wATile);
          const uint64_t db = sw128_kmajor_desc(sm0 + s * wBTile);
          const uint32_t sf = tmem_base + (uint32_t)(wSfCol0 + 16 * s);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // Scale ids (bits 4-5 for B, 29-30 for A) pick byte k of the scale words.
            umma_mxf8(tmem_base, da + 2 * k, db + 2 * k, kIdesc0 | ((uint32_t)k << 4) | ((uint32_t)k << 29), sf,
                      sf + 8, (kb | k) ? 1u : 0u);
          }
          issued = true;
          umma_commit(empty(s));
        }
        if (!ok) break;
        umma_commit(tfull_bar);
      }
      if (!ok && issued) {
        umma_commit(drain_bar);
        drain_wait(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quarter this warp may read
    const int hh = (warp - wEpiWarp0) >> 2;    // which 128 accumulator columns
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(tfull_bar, (uint32_t)local & 1u, abort_flag, p.status,
                               MOE_DEV_TIMEOUT_EPILOGUE, p.limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      // Accumulator columns of this warp: GEMM-1 gate 64 (two blocks of 32), then
      // up 64; GEMM-2 128 consecutive y columns.
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(hh * 128);
      uint32_t g0[32], g1[32], u0[32], u1[32];
      tmem_ld_32x32b_x32(tb, g0);
      tmem_ld_32x32b_x32(tb + 32, g1);
      tmem_ld_32x32b_x32(tb + 64, u0);
      tmem_ld_32x32b_x32(tb + 96, u1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar);  // the MMA may overwrite the accumulator now
      const TileInfo ti = decode_tile_s<128>(p.G, tile_start, row_start, tile);
      const int r = ti.tt * 128 + q * 32 + lane;
      if (MODE == 1) {
        // y leaves through this warp's 2 KB staging block, 16 columns at a
        // time: each lane writes its row's four 16-byte chunks (chunk c of row
        // i at position c ^ ((i >> 1) & 3), so neither side has bank
        // conflicts), then every store instruction writes eight rows' 64-byte
        // segments (four lanes a row) instead of 16 bytes in each of 32 rows.
        float* stg = y_stage + (warp - wEpiWarp0) * wStgWarp;
        const int r0 = ti.tt * 128 + q * 32;  // this warp's first row within the group
        float* ycol = static_cast<float*>(p.out) + (size_t)ti.row0 * p.N + ti.wt * kCols + hh * 128;
        auto put = [&](const uint32_t (&v)[32], int c0) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<float4*>(stg + lane * 16 + ((c ^ ((lane >> 1) & 3)) << 2)) =
                  make_float4(__uint_as_float(v[16 * b + 4 * c]), __uint_as_float(v[16 * b + 4 * c + 1]),
                              __uint_as_float(v[16 * b + 4 * c + 2]), __uint_as_float(v[16 * b + 4 * c + 3]));
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = (lane >> 2) + 8 * k, c = lane & 3;
              const float4 val = *reinterpret_cast<const float4*>(stg + i * 16 + ((c ^ ((i >> 1) & 3)) << 2));
              if (r0 + i < ti.nrows)
                *reinterpret_cast<float4*>(ycol + (size_t)(r0 + i) * p.N + c0 + 16 * b + 4 * c) = val;
            }
            __syncwarp();
          }
        };
        put(g0, 0);
        put(g1, 32);
        put(u0, 64);
        put(u1, 96);
      } else if (r < ti.nrows) {
        const long long a_blk = tile_start[ti.g] / n_wt + ti.tt;
        uint8_t* h_atoms = p.out_scale + a_blk * (p.N / 128) * kAtomBytes;
        const int col = ti.wt * 128 + hh * 64;
        uint8_t* hrow = static_cast<uint8_t*>(p.out) + (size_t)(ti.row0 + r) * p.N + col;
        uint8_t* srow = h_atoms + (size_t)(col / 128) * kAtomBytes;
        const int j0 = (col / 32) & 3;
        store_h_block(g0, u0, hrow, srow + atom_byte(q * 32 + lane, j0));
        store_h_block(g1, u1, hrow + 32, srow + atom_byte(q * 32 + lane, j0 + 1));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, wTmemCols);
  }
}

template <int MODE, bool W4>
cudaError_t run_gemm_mx_wide(const GroupedGemmArgs& a, cudaStream_t s) {
  if (a.rows == 0 || a.G == 0) return cudaSuccess;
  if (a.H % 128 || a.I % 128 || a.G > wMaxGroups || (MODE == 1 && a.H % 256)) return cudaErrorInvalidValue;
  const int G = a.offsets ? a.G : 1;
  const int Kdim = MODE == 0 ? a.H : a.I;
  const int N = MODE == 0 ? a.I : a.H;
  const void* act = MODE == 0 ? a.a : a.h;
  CUtensorMap m_act, m_w0, m_w1;
  bool maps_ok = make_tmap_u8(&m_act, act, Kdim, a.rows, 128);
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
  const long long max_tiles = n_wt * ((a.rows + 127) / 128 + G);
  const int grid = (int)(max_tiles < a.num_sms ? max_tiles : a.num_sms);
  grouped_gemm_mx_wide_kernel<MODE, W4><<<grid, wThreads, wSmemFor<MODE>(), s>>>(m_act, m_w0, m_w1, p);
  return cudaGetLastError();
}

}  // namespace

bool gemm_mx_wide_supported(const GroupedGemmArgs& a, int mode) {
  return (a.offsets ? a.G : 1) <= wMaxGroups && (mode == 0 || a.H % 256 == 0);
}

cudaError_t gemm_mx_wide_prepare_device() {
  const cudaError_t errs[] = {
      cudaFuncSetAttribute(grouped_gemm_mx_wide_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, wSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_wide_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, wSmem),
      cudaFuncSetAttribute(grouped_gemm_mx_wide_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           wSmemFor<1>()),
      cudaFuncSetAttribute(grouped_gemm_mx_wide_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           wSmemFor<1>())};
  for (cudaError_t e : errs)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_gemm_mx_wide_gate_up(const GroupedGemmArgs& a, cudaStream_t s) {
  return a.w4 ? run_gemm_mx_wide<0, true>(a, s) : run_gemm_mx_wide<0, false>(a, s);
}

cudaError_t launch_gemm_mx_wide_down(const GroupedGemmArgs& a, cudaStream_t s) {
  return a.w4 ? run_gemm_mx_wide<1, true>(a, s) : run_gemm_mx_wide<1, false>(a, s);
}

}  // namespace moe
