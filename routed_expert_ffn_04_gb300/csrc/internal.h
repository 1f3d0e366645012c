// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units. Host-side only; nothing here is exported.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/moe.h"

namespace moe {

// Handle accessors for translation units other than api.cu.
int handle_device(moe_handle_t h);
int* handle_status_word(moe_handle_t h);

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Both MX dtypes carry E4M3 activations (1 byte per element) with one E8M0
// scale per 32 elements; they differ only in the routed experts' weights.
inline bool is_mx_dtype(int dtype) { return dtype == MOE_MXFP8_E4M3 || dtype == MOE_MXFP4_W4A8; }

// ---- routing (route.cu)
cudaError_t launch_route(const float* logits, int T, int E, int K, float scaling, int route_norm,
                         int32_t* topk_idx, float* topk_w, cudaStream_t s);

// ---- gating + routing for few tokens (gate.cu): CUDA-core split-K in one
// cluster launch, E <= 256, T <= kGateSmallMaxT. x [T, H] and w_router
// [E, H] bf16; logits [T, E] fp32 out (nullable).
constexpr int kGateSmallMaxT = 256;
bool gate_route_small_fits(int T, int H, int E);
cudaError_t gate_small_prepare_device();
cudaError_t launch_gate_route_small(const void* x, const void* w_router, int T, int H, int E,
                                    int K, float scaling, int route_norm, float* logits,
                                    int32_t* topk_idx, float* topk_w, cudaStream_t s);

// ---- permutation (permute.cu)
size_t permute_scratch_bytes(int TK, int E);
// Opt the cluster permutation into its dynamic shared memory (once per device).
cudaError_t permute_prepare_device();
// counts [E], offsets [E+1], perm_src / flat_to_perm [TK]; tile_offsets
// (nullable) [E+1]: the first 128-row tile of each expert. scratch is used
// only above the single-launch sizes (more than 262144 pairs).
cudaError_t launch_permute_index(const int32_t* topk_idx, int TK, int E, void* scratch,
                                 int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                                 int32_t* perm_src, int32_t* flat_to_perm, int* status,
                                 cudaStream_t s);
// dst[r, :] = src[perm_src[r] / K, :] for r < TK; rows are row_bytes long
// (a multiple of 16). A perm_src entry outside [0, TK) gives a zero row.
// x_perm[flat_to_perm[t*K+k]] = x[t] for every token t and slot k: each
// source row read once (row_bytes a multiple of 4).
cudaError_t launch_scatter_rows(const void* src, int T, int row_bytes, const int32_t* flat_to_perm,
                                int K, int TK, void* dst, int* status, cudaStream_t s);
// MX rows: x_q [T, H] E4M3 codes -> x_perm [TK, H], and the row-major scales
// x_scale [T, H/32] into the scale atoms of the permuted rows (by expert tile,
// tile_offsets from launch_permute_index). H % 128 == 0.
cudaError_t launch_scatter_rows_mx(const uint8_t* x_q, const uint8_t* x_scale, int T, int H,
                                   const int32_t* flat_to_perm, const int32_t* topk_idx,
                                   const int32_t* offsets, const int32_t* tile_offsets, int K, int TK,
                                   int E, uint8_t* x_perm, uint8_t* atoms, int* status,
                                   cudaStream_t s);

// ---- grouped GEMM (gemm.cu)
// kModePair: weights as the M = 256 rows of an MMA spread over a CTA pair
// (gemm_pair.cu), tokens as N.
enum GemmMode { kModeAuto = 0, kModeWeightsM = 1, kModeTokensM = 2, kModePair = 3 };

struct GroupedGemmArgs {
  int G;                   // number of groups
  const int32_t* offsets;  // [G+1] device, or nullptr: one group of `rows`
  int rows;                // activation rows
  int H, I;                // hidden, intermediate
  const void* a;           // [rows, H] bf16
  const void* w_gate;      // [G, I, H] bf16
  const void* w_up;        // [G, I, H] bf16
  const void* w_down;      // [G, H, I] bf16
  void* h;                 // [rows, I] bf16 (intermediate)
  float* y;                // [rows, H] fp32
  int32_t* topk_idx;       // gating: routing outputs [rows, topk]
  float* topk_w;
  int topk;
  float scaling;
  int route_norm;
  int mode;                // GemmMode
  // MXFP8 (gemm_mx.cu): a / h hold E4M3 codes and their scales are atoms by
  // token tile of each group; s_gate the gate/up atoms, s_down the down atoms.
  // w4: the weights are packed E2M1 (two per byte, MXFP4) instead of E4M3.
  const uint8_t* a_scale;
  uint8_t* h_scale;
  const uint8_t* s_gate;
  const uint8_t* s_down;
  int w4;
  // MX GEMM tiling: 0 auto, 1 = 128 weight rows (gemm_mx.cu), 2 = 256 rows
  // (gemm_mx_wide.cu), 3 = weights as M (gemm_mx_swap.cu).
  int mx_tile;
  // bf16 GEMM-1, tokens-as-M tiling: gather the A rows from x instead of
  // reading a: row r is token gather_src[r] / gather_k of gather_x [T, H]
  // (nullptr: read a).
  const int32_t* gather_src;
  int gather_k;
  const void* gather_x;
  // bf16 only: the shared expert's [I, H], [I, H], [H, I] weights, run as the
  // last of the G groups (nullptr: every group uses w_gate / w_up / w_down).
  const void* shared_w_gate;
  const void* shared_w_up;
  const void* shared_w_down;
  int num_sms;
  int* status;
  uint64_t wait_limit_ns;
};
bool gemm_init_driver();  // resolves cuTensorMapEncodeTiled; false if unavailable
// Opt the GEMM kernels into their dynamic shared memory on the current device
// (once per device, outside any stream capture).
cudaError_t gemm_prepare_device();
// 2-D fp32 tensor map [outer, inner] for bulk stores of 32 x 32 blocks from a
// 128-byte-swizzled shared-memory buffer (inner % 32 == 0).
bool make_tmap_f32_store(CUtensorMap* m, void* ptr, uint64_t inner, uint64_t outer);
// 2-D bf16 tensor map [outer, inner], box {64 elements, box_rows}, 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows);
// 2-D uint8 tensor map [outer, inner], box {128 bytes, box_rows}, 128-byte swizzle.
bool make_tmap_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_rows);
// Tensor map of packed E2M1 weights in tile order (moe_tile_mxfp4_weights),
// read as rows64 rows of 128 elements (64 bytes each, contiguous; ptr 32-byte
// aligned), box {128 elements, box_rows}: each 16 codes (8 bytes) land in the
// low half of a 16-byte shared-memory slot, 128-byte swizzle, the operand
// layout of kind::mxf8f6f4 for E2M1. A box's transaction count is its global
// bytes (64 per row). The row of block (t, kb), row r is (t * nk + kb) * R + r,
// R = 128 (one matrix) or 256 (a gate/up pair).
bool make_tmap_e2m1(CUtensorMap* m, const void* ptr, uint64_t rows64, uint32_t box_rows);
// Native MXFP8 grouped GEMM (gemm_mx.cu): block-scaled tcgen05 MMA, E4M3
// activations (a + a_scale; GEMM-2 reads h + h_scale) and weights.
cudaError_t gemm_mx_prepare_device();
cudaError_t launch_gemm_mx_gate_up(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_mx_down(const GroupedGemmArgs& a, cudaStream_t s);
// MX GEMMs with 256 weight rows per MMA (gemm_mx_wide.cu): up to 512 groups;
// GEMM-2 (mode 1) needs H % 256 == 0.
bool gemm_mx_wide_supported(const GroupedGemmArgs& a, int mode);
cudaError_t gemm_mx_wide_prepare_device();
cudaError_t launch_gemm_mx_wide_gate_up(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_mx_wide_down(const GroupedGemmArgs& a, cudaStream_t s);
// MX GEMMs with the weights as M (gemm_mx_swap.cu): 256 weight rows against
// up to 64 token rows per tile; up to 512 groups; GEMM-2 needs H % 256 == 0.
bool gemm_mx_swap_supported(const GroupedGemmArgs& a, int mode);
cudaError_t gemm_mx_swap_prepare_device();
cudaError_t launch_gemm_mx_swap_gate_up(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_mx_swap_down(const GroupedGemmArgs& a, cudaStream_t s);
// The tiling launch_gemm_gate_up / launch_gemm_down will use (GemmMode).
int gemm_pick_mode(const GroupedGemmArgs& a);
cudaError_t launch_gemm_gate_up(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_down(const GroupedGemmArgs& a, cudaStream_t s);
// CTA-pair bf16 grouped GEMM (gemm_pair.cu); not for a folded shared expert.
bool gemm_pair_supported(const GroupedGemmArgs& a);
cudaError_t gemm_pair_prepare_device();
cudaError_t launch_gemm_pair_gate_up(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_pair_down(const GroupedGemmArgs& a, cudaStream_t s);
// Gating GEMM (one group, E <= 256) with routing in its epilogue: a.h = x
// [rows, a.I], a.w_down = router weights [a.H = E, a.I], a.y = logits out
// (nullable), routing into a.topk_idx / a.topk_w.
cudaError_t launch_gate_route(const GroupedGemmArgs& a, cudaStream_t s);

// ---- combine (combine.cu)
cudaError_t launch_combine(const float* y_perm, const float* topk_w, const int32_t* flat_to_perm,
                           const float* shared_out, int T, int K, int H, void* out, int* status,
                           cudaStream_t s);

// ---- MX quantiser (mxquant.cu)
// q / scale / atoms may each be null. scale: row-major [rows, cols/32];
// atoms: the scale atoms of the rows as one group (cols % 128 == 0; the rows
// of the last 128-row block past `rows` are left untouched).
cudaError_t launch_mx_quantize(const void* in_bf16, int64_t rows, int cols, uint8_t* q,
                               uint8_t* scale, uint8_t* atoms, cudaStream_t s);

// MXFP4: q [rows, cols/2] packed E2M1 codes (element 2j in the low nibble),
// scale [rows, cols/32] row-major.
cudaError_t launch_mx4_quantize(const void* in_bf16, int64_t rows, int cols, uint8_t* q,
                                uint8_t* scale, cudaStream_t s);

// ---- scale atoms (mxpack.cu; layout in mx_layout.cuh)
// Row-major E8M0 scales [rows, cols/32] -> atoms. s1 == nullptr: the atoms
// of s0 (rows % 128 == 0). Else gate (s0) and up (s1) interleaved per 64 rows
// (rows % 64 == 0), 2 * rows atom-matrix rows. cols % 128 == 0.
// Packed E2M1 [rows, cols/2] (a gate/up pair with q1) -> the tile order of
// moe_tile_mxfp4_weights.
cudaError_t launch_tile_e2m1(const uint8_t* q0, const uint8_t* q1, int64_t rows, int cols, uint8_t* dst,
                             cudaStream_t s);
cudaError_t launch_pack_weight_scales(const uint8_t* s0, const uint8_t* s1, int64_t rows, int cols,
                                      uint8_t* out, cudaStream_t s);
// Activation scales [src_rows, cols/32] -> atoms by token tile of each group
// (offsets [G+1], or nullptr for one group of `rows`). Row j of group g takes
// the scales of src row perm_src[offsets[g] + j] / K (nullptr: offsets[g] + j).
cudaError_t launch_gather_scale_atoms(const uint8_t* src, int src_rows, int cols,
                                      const int32_t* perm_src, int K, const int32_t* offsets,
                                      int G, int rows, uint8_t* out, int* status, cudaStream_t s);
// Bytes of activation atoms for `rows` rows in at most `groups` groups.
size_t scale_atom_bytes(int64_t rows, int groups, int cols);
// ---- self-test of the bounded wait (gemm.cu)
cudaError_t launch_selftest_wait(int* status, uint64_t limit_ns, cudaStream_t s);

}  // namespace moe
