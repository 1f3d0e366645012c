/*
 * moe.h - C ABI of the GB300 (sm_103a) sigmoid-routed top-k MoE FFN layer.
 *
 * The layer (forward pass) is the MoE block of the Hy3 / Hy4 /
 * HunyuanImage-3.0 models:
 *   out[t] = sum_k w[t,k] * FFN_{e(t,k)}(x[t]) + FFN_shared(x[t])
 * with FFN(x) = W_down (silu(W_gate x) * (W_up x)) and (e, w) from sigmoid
 * top-k routing with route_norm and router_scaling_factor.
 *
 * Passages that define it (page titles):
 *   [Hy3]  "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战"
 *          section 一: 192 routed experts, top-8 sigmoid routing, 1 shared
 *          expert, expert intermediate 1536, hidden 4096,
 *          router_scaling_factor=2.826, route_norm=True.
 *          section 8.5: the main stream runs gating, then the routed path
 *          (InitRouting -> grouped GMM -> FinalizeRouting), then the combine
 *          add; the shared expert runs on a second stream that starts after
 *          gating and is joined before the add.
 *          section 8.2: routed and shared Linears in W8A8 MXFP8.
 *   [HyI3] "HunyuanImage-3.0 MoE 多流变体实战", 源码级实现拆解 §1-§3:
 *          a side stream created once and passed in; input_ready_event
 *          recorded on the main stream and waited on by the side stream;
 *          mlp_done_event recorded on the side stream and waited on by the
 *          main stream; output = hidden_states_mlp + combined_output.
 *
 * Conventions for every entry point:
 *   - Pointers marked (device) are CUDA device pointers; the caller owns all
 *     buffers. No entry point allocates device memory per call; scratch comes
 *     from a caller-provided workspace whose size the *_workspace_size calls
 *     return. moe_create allocates a 64-byte device status word once.
 *   - Every device pointer must be 16-byte aligned (MOE_ERR_INVALID_ARG).
 *   - Matrices are dense row-major. Weights are K-major: the reduction axis
 *     is the last (contiguous) one.
 *   - Calls are asynchronous on the given stream(s) and never synchronise
 *     the host, except moe_get_device_status, moe_read_stage_times and
 *     moe_layer_forward_host, which say so.
 *   - Argument errors are returned before any launch. A failed launch
 *     returns MOE_ERR_CUDA. A device-side wait that gives up (a bounded
 *     spin, about 2 s) records a code in the handle's status word, which
 *     moe_get_device_status reports; outputs of that call are undefined.
 *   - A handle is bound to one device and is not thread-safe; use one
 *     handle per concurrently used stream pair.
 *   - Streams are cudaStream_t values passed as void*; NULL is the legacy
 *     default stream.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_API __attribute__((visibility("default")))

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or config */
  MOE_ERR_UNSUPPORTED = 2,   /* valid request the library does not handle */
  MOE_ERR_WORKSPACE = 3,     /* workspace smaller than *_workspace_size */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_TIMEOUT = 5 /* a device-side bounded wait gave up */
} moe_status_t;

typedef enum {
  MOE_BF16 = 0,       /* bf16 operands, fp32 accumulation */
  MOE_MXFP8_E4M3 = 1, /* E4M3 elements + one E8M0 scale per 32 along K */
  MOE_MXFP4_W4A8 = 2  /* W4A8 ([Hy3] section 8.2): routed-expert weights E2M1 +
                         E8M0/32 (MXFP4), activations MXFP8, shared expert W8A8 */
} moe_dtype_t;

/* Layer shape. T tokens, H hidden, E routed experts, K experts per token,
 * I routed-expert intermediate size, I_shared shared-expert intermediate size
 * (0 = no shared expert). scaling = router_scaling_factor ([Hy3] section 一:
 * 2.826); route_norm != 0 divides the K sigmoid scores by their sum.
 * Limits: 1 <= K <= min(E, 32), E <= 1024, H % 64 == 0, I % 64 == 0,
 * I_shared % 64 == 0 (MXFP8: H, I, I_shared % 128 == 0), T * K < 2^31,
 * T*K*max(H,I) < 2^40. */
typedef struct {
  int T, H, E, K, I, I_shared;
  float scaling;
  int route_norm;
  moe_dtype_t dtype;
} moe_config_t;

/* Layer weights (device). bf16 mode: w_* are bf16, s_* ignored.
 *   w_gate, w_up: [E, I, H]     w_down: [E, H, I]
 *   ws_gate, ws_up: [I_shared, H]   ws_down: [H, I_shared]  (NULL if I_shared == 0)
 * MXFP8 mode: w_* are E4M3 codes (uint8) and the E8M0 scales (one per 32
 * consecutive elements of a row) are given as scale atoms, the layout the
 * block-scaled tensor cores read, written by moe_pack_mx_scales:
 *   s_gate  = atoms of gate and up together (moe_pack_mx_scales(gate, up)),
 *   s_down  = atoms of down (moe_pack_mx_scales(down, NULL)),
 *   s_up    unused (NULL); ss_gate, ss_up, ss_down the same for the shared
 *   expert. Every scale pointer 16-byte aligned.
 * MXFP4_W4A8 mode: as MXFP8, except that the routed weights are packed E2M1
 *   codes (two per byte, element 2j in the low nibble; moe_quantize_mxfp4) in
 *   tile order: w_gate = moe_tile_mxfp4_weights(gate, up) of the [E*I, H]
 *   gate and up codes together, w_up unused (NULL), w_down =
 *   moe_tile_mxfp4_weights(down, NULL) of [E*H, I]; 32-byte aligned. Their
 *   scales and the shared expert (E4M3 + atoms) are as in MXFP8 mode. */
typedef struct {
  const void *w_gate, *w_up, *w_down;
  const uint8_t *s_gate, *s_up, *s_down;
  const void *ws_gate, *ws_up, *ws_down;
  const uint8_t *ss_gate, *ss_up, *ss_down;
} moe_weights_t;

typedef struct moe_handle* moe_handle_t;
typedef void* moe_stream_t; /* a cudaStream_t */

/* Options for moe_set_option. */
typedef enum {
  /* Grouped GEMM tiling: 0 = automatic (default: 1 up to 48 rows per group
   * on average, 2 above), 1 = weight rows fill the 128-row MMA tile and
   * tokens form N (small token counts per expert), 2 = tokens fill the
   * 128-row MMA tile, 3 = weight rows fill a 256-row MMA spread over a pair
   * of SMs and up to 128 (GEMM-1) or 256 (GEMM-2) tokens form N (large token
   * counts per expert; bf16 only, and not with MOE_OPT_SHARED_FOLD, where 2
   * is used instead). MX layers use their own kernels whatever the value. */
  MOE_OPT_GEMM_MODE = 0,
  /* 1 = record CUDA events between the stages of moe_layer_forward so
   * moe_read_stage_times can report per-stage device time. Default 0. */
  MOE_OPT_STAGE_TIMING = 1,
  /* Device wait limit in microseconds for bounded spins (default 2000000). */
  MOE_OPT_WAIT_LIMIT_US = 2,
  /* 1 = run the shared expert as one more group of the routed grouped GEMMs
   * instead of on the side stream (bf16 layers with I_shared == I and
   * E <= 1023; otherwise ignored). The result is the same; which is faster
   * depends on the shape. Default 0 (side stream). */
  MOE_OPT_SHARED_FOLD = 3,
  /* SMs given to the shared expert while it runs on the side stream; the
   * routed GEMMs' persistent grids take the rest. 0 = no split (default):
   * both streams' GEMMs size their grids to every SM, and the shared
   * kernels fill the SMs that routing and permutation leave idle (no fixed
   * split measured faster on the decode, MX, skewed or prefill workloads).
   * k > 0 = k SMs (at most half). The result is the same either way. */
  MOE_OPT_SHARED_SMS = 4,
  /* 1 (default) = in bf16 layers whose routed GEMM-1 takes the tokens-as-M
   * tiling (more than 48 rows per expert on average, or mode 2), the GEMM-1
   * loads its A rows straight from x through perm_src (InitRouting's row
   * gather fused into the grouped GEMM) and x_perm is not written; 0 = the
   * permutation writes x_perm and GEMM-1 reads it. The result is the same. */
  MOE_OPT_GATHER_A = 5,
  /* Tiling of the MX (MXFP8, W4A8) grouped GEMMs: 0 = automatic (default:
   * 3 when the GEMM has at most 48 rows per expert on average, as in decode;
   * otherwise 2, except 1 for a single group with E4M3 weights such as the
   * shared expert), 1 = 128 token rows x 128
   * weight rows per MMA (GEMM-1 gate 64 + up 64; double-buffered
   * accumulators), 2 = 128 token rows x 256 weight rows (GEMM-1 gate 128 + up
   * 128; GEMM-2 when H % 256 == 0; one accumulator), 3 = weights as M: 256
   * weight rows as two 128-row MMAs against up to 64 token rows of one
   * expert (GEMM-2 when H % 256 == 0; at most 512 groups; else 2 for E2M1
   * weights, 1 for E4M3). The result is the same up to fp32 summation order. */
  MOE_OPT_MX_TILE = 6
} moe_option_t;

/* Stage indices reported by moe_read_stage_times. */
enum {
  MOE_STAGE_ROUTE = 0,        /* sigmoid top-k routing kernel            */
  MOE_STAGE_PERMUTE = 1,      /* histogram, scan, scatter, row gather    */
  MOE_STAGE_GEMM_GATE_UP = 2, /* routed grouped GEMM-1 + SwiGLU epilogue */
  MOE_STAGE_GEMM_DOWN = 3,    /* routed grouped GEMM-2                   */
  MOE_STAGE_COMBINE = 4,      /* join with the shared stream + combine   */
  MOE_STAGE_SHARED = 5,       /* shared expert on its stream             */
  MOE_STAGE_TOTAL = 6,        /* whole call on the main stream           */
  MOE_NUM_STAGES = 7
};

/* Create a handle on `device`: records the SM count, resolves the TMA
 * descriptor encoder, sets the kernels' shared-memory limits on the device,
 * allocates the device status word and two events. Returns MOE_ERR_CUDA if
 * the device is unusable. After this, moe_layer_forward makes no allocation
 * or device-attribute call, so a call (with stage timing off) can be
 * captured into a CUDA graph on `main`, the side stream joining through the
 * handle's two events. */
MOE_API moe_status_t moe_create(int device, moe_handle_t* out);
MOE_API moe_status_t moe_destroy(moe_handle_t h);
MOE_API const char* moe_status_string(moe_status_t s);
MOE_API moe_status_t moe_set_option(moe_handle_t h, moe_option_t opt, int value);

/* Workspace bytes moe_layer_forward / moe_layer_forward_host need for cfg
 * (host-only, no GPU needed). */
MOE_API moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Step 1, routing ([Hy3] section 一; the gating result is the input).
 * logits (device): [T, E] fp32. Per token, the K experts with the largest
 * fp32 logits, in descending logit order, equal logits -> lower id first
 * (+0 and -0 are equal; NaN ranks below every number).
 * topk_w[t,k] = scaling * sigma(l_k) / (route_norm ? sum_j sigma(l_j) : 1).
 * topk_idx (device): [T, K] int32 out. topk_w (device): [T, K] fp32 out. */
MOE_API moe_status_t moe_route(moe_handle_t h, const moe_config_t* cfg, const float* logits,
                               int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/* Scratch bytes moe_permute needs (host-only). */
MOE_API moe_status_t moe_permute_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Step 2, InitRouting ([Hy3] sections 8.1, 8.5): stable counting sort of the
 * T*K (token, slot) pairs (flat index f = t*K + k) by expert id, then a row
 * gather. Outputs (device): counts [E], offsets [E+1] (exclusive scan),
 * perm_src [T*K] (permuted row -> f), flat_to_perm [T*K] (its inverse),
 * x_perm [T*K, H] = x[perm_src[r] / K]. Rows of one expert keep ascending f.
 * x (device): [T, H] bf16; MXFP8 mode: E4M3 codes with x_scale [T, H/32]
 * and x_perm_scale [T*K, H/32] (else both ignored). An expert id outside
 * [0, E) is skipped and recorded in the device status word. */
MOE_API moe_status_t moe_permute(moe_handle_t h, const moe_config_t* cfg, const void* x,
                                 const uint8_t* x_scale, const int32_t* topk_idx, int32_t* counts,
                                 int32_t* offsets, int32_t* perm_src, int32_t* flat_to_perm,
                                 void* x_perm, uint8_t* x_perm_scale, void* ws, size_t ws_bytes,
                                 moe_stream_t stream);

/* Scratch bytes moe_grouped_swiglu_gemm needs for `rows` rows in
 * `num_groups` groups: the [rows, I] intermediate (bf16, or MXFP8 E4M3 codes
 * plus the scale atoms of h and of `a`, one atom row-block per 128 rows of
 * each group). */
MOE_API moe_status_t moe_grouped_gemm_workspace_size(int rows, int num_groups, int H, int I,
                                                     moe_dtype_t dtype, size_t* bytes);

/* Step 3, the grouped expert GEMM with SwiGLU (the grouped GMM of [Hy3]
 * section 8.5): for each group g, rows offsets[g] .. offsets[g+1]-1 of `a`:
 *   h = silu(a W_gate[g]^T) * (a W_up[g]^T)   (fp32 accumulate, h stored bf16
 *                                              or, in MXFP8 mode, re-quantised)
 *   y = h W_down[g]^T                          (fp32 accumulate, stored fp32)
 * a (device): [rows, H] bf16 (MXFP8: E4M3 codes + a_scale [rows, H/32] E8M0,
 *   row-major).
 * MXFP8: w_* are E4M3 codes; s_gate = moe_pack_mx_scales(gate, up) atoms of
 *   the [num_groups*I, H/32] gate and up scales, s_down =
 *   moe_pack_mx_scales(down, NULL) atoms of the [num_groups*H, I/32] down
 *   scales, s_up unused. h is rounded to MXFP8 (blocks of 32 along I) before
 *   GEMM-2, as the W8A8 path quantises every Linear input ([Hy3] section
 *   8.2). Operands and scales go to the block-scaled tensor cores as stored.
 *   H % 128 == 0, I % 128 == 0.
 * MXFP4_W4A8: w_gate = moe_tile_mxfp4_weights(gate, up) of the packed E2M1
 *   codes of [num_groups*I, H] gate and up weights, w_up unused, w_down =
 *   moe_tile_mxfp4_weights(down, NULL) of [num_groups*H, I]; 32-byte aligned;
 *   scales and a as in MXFP8.
 * offsets (device): [num_groups + 1] int32, non-decreasing, offsets[0] = 0,
 *   offsets[num_groups] <= rows; NULL means one group of all rows (a dense
 *   SwiGLU MLP, used for the shared expert).
 * w_gate, w_up: [num_groups, I, H]; w_down: [num_groups, H, I] (device).
 * y (device): [rows, H] fp32 out; rows outside every group are not written.
 * Limits: num_groups <= 1024, H % 64 == 0, I % 64 == 0. */
MOE_API moe_status_t moe_grouped_swiglu_gemm(moe_handle_t h, int num_groups, int rows, int H,
                                             int I, moe_dtype_t dtype, const void* a,
                                             const uint8_t* a_scale, const int32_t* offsets,
                                             const void* w_gate, const void* w_up,
                                             const void* w_down, const uint8_t* s_gate,
                                             const uint8_t* s_up, const uint8_t* s_down, float* y,
                                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* Step 4, FinalizeRouting + shared add ([Hy3] section 8.5 "combine 相加";
 * [HyI3] §3 output = hidden_states_mlp + combined_output):
 *   out[t] = bf16_rne( sum_{k=0..K-1} topk_w[t,k] * y_perm[flat_to_perm[t*K+k]]
 *                      + shared_out[t] )
 * summed in fp32 in that order and rounded once.
 * y_perm (device): [T*K, H] fp32; topk_w: [T, K] fp32; flat_to_perm: [T*K];
 * shared_out (device, nullable): [T, H] fp32; out (device): [T, H] bf16.
 * A flat_to_perm entry of -1 (a pair moe_permute dropped for an expert id out
 * of range) adds nothing and is not reported again; any other entry outside
 * [0, T*K) adds nothing and records MOE_DEV_BAD_PERM_INDEX. */
MOE_API moe_status_t moe_combine(moe_handle_t h, const moe_config_t* cfg, const float* y_perm,
                                 const float* topk_w, const int32_t* flat_to_perm,
                                 const float* shared_out, void* out, moe_stream_t stream);

/* MXFP8 quantisation of a bf16 matrix along its rows (npu_dynamic_mx_quant in
 * [Hy3] section 六; rule of the OCP MX v1.0 spec): per block of 32, scale
 * X = 2^(floor(log2 amax) - 8) stored as E8M0, elements RNE(v / X) to E4M3
 * saturating at +-448; an all-zero block gets scale code 0.
 * in (device): [rows, cols] bf16; q (device): [rows, cols] uint8 out;
 * scale (device): [rows, cols/32] uint8 out. cols % 32 == 0. */
MOE_API moe_status_t moe_quantize_mxfp8(moe_handle_t h, const void* in_bf16, int64_t rows,
                                        int cols, uint8_t* q, uint8_t* scale, moe_stream_t stream);

/* MXFP4 quantisation of a bf16 matrix along its rows (the W4A8 routed-expert
 * weights of [Hy3] section 8.2; rule of the OCP MX v1.0 spec with E2M1
 * elements): per block of 32, scale X = 2^(floor(log2 amax) - 2) stored as
 * E8M0, elements rounded to nearest-even on the E2M1 grid (0, 0.5, 1, 1.5, 2,
 * 3, 4, 6) saturating at +-6; an all-zero block gets scale code 0.
 * in (device): [rows, cols] bf16; q (device): [rows, cols/2] uint8 out, two
 * codes per byte (element 2j in the low nibble); scale (device): [rows,
 * cols/32] uint8 out. cols % 32 == 0. */
MOE_API moe_status_t moe_quantize_mxfp4(moe_handle_t h, const void* in_bf16, int64_t rows,
                                        int cols, uint8_t* q, uint8_t* scale, moe_stream_t stream);

/* Tile order of packed E2M1 weights, the form the W4A8 grouped GEMMs read
 * (a one-time weight step, like the page's weight conversion, section 五
 * "转换权重", which derives the MXFP4 routed-expert weights for the MoE GMM).
 * q0, q1 (device): [rows, cols/2] packed E2M1 as moe_quantize_mxfp4 writes it.
 * tiled (device): one contiguous block per 128-row block t and 128-element K
 * block kb (K blocks of a row block consecutive, row blocks in order), the
 * rows of 64 bytes each:
 *   q1 == NULL (w_down): 8 KB at byte 8192 (t * (cols/128) + kb), rows
 *     128 t .. 128 t + 127 of q0; tiled holds rows * cols/2 bytes.
 *   q1 != NULL (w_gate = q0, w_up = q1, packed together as
 *     moe_pack_mx_scales packs their scales): 16 KB at byte 16384 (t *
 *     (cols/128) + kb): rows 0-63 of the block from q0, then from q1, then
 *     rows 64-127 from q0, then from q1; tiled holds 2 * rows * cols/2 bytes.
 * One such block is exactly what one TMA load of the W4A8 GEMM-1 (a pair
 * block) or GEMM-2 (a w_down block) fetches per K stage, so a stage is one
 * contiguous read and one copy instruction. rows % 128 == 0, cols % 128 == 0,
 * tiled distinct from q0 and q1, all 16-byte aligned. */
MOE_API moe_status_t moe_tile_mxfp4_weights(moe_handle_t h, const uint8_t* q0, const uint8_t* q1, int64_t rows,
                                            int cols, uint8_t* tiled, moe_stream_t stream);

/* Scale atoms for the block-scaled MXFP8 GEMM from row-major E8M0 scales
 * (as moe_quantize_mxfp8 writes them). An atom holds the scales of 128 rows
 * x 128 elements (4 per row) in 512 bytes: row r of the block, K-block j at
 * byte 16 (r % 32) + 4 (r / 32) + j; the atoms of a matrix follow each other
 * row-block major (128-row block b, K-block a at atom b * cols/128 + a).
 * scale1 == NULL: atoms of scale0 [rows, cols/32], rows % 128 == 0.
 * scale1 != NULL: gate (scale0) and up (scale1) scales, each [rows, cols/32]
 *   with rows % 64 == 0, interleaved per 64 rows (gate rows 0-63, up rows
 *   0-63, gate rows 64-127, ...) into a 2*rows-row atom matrix: the row order
 *   of one GEMM-1 tile. Use it for the per-expert [E*I] gate/up pair.
 * cols % 128 == 0. atoms (device): rows * cols / 32 bytes (twice that with
 * scale1). Pointers 16-byte aligned. Packing is a one-time weight step. */
MOE_API moe_status_t moe_pack_mx_scales(moe_handle_t h, const uint8_t* scale0,
                                        const uint8_t* scale1, int64_t rows, int cols,
                                        uint8_t* atoms, moe_stream_t stream);

/* The whole layer, steps 1-4 plus the shared expert, with the two-stream
 * orchestration of [Hy3] section 8.5 / [HyI3] §3: an event recorded on
 * `main` at entry is waited on by `side`, which runs the shared expert and
 * records a second event that `main` waits on before the combine.
 * side == NULL runs the shared expert on `main` before the routed path.
 * x (device): [T, H] bf16. In the MX modes (weights then E4M3 / E2M1 codes +
 * scale atoms, for example moe_quantize_mxfp8 on the bf16 weights then
 * moe_pack_mx_scales):
 *   x_scale_or_null == NULL: x is bf16 and is quantised inside, per call,
 *     with the rule of moe_quantize_mxfp8;
 *   x_scale_or_null != NULL: x already holds E4M3 codes [T, H] (uint8) and
 *     x_scale_or_null their E8M0 scales [T, H/32], row-major, as
 *     moe_quantize_mxfp8 writes them; nothing is re-quantised.
 * bf16 mode: x_scale_or_null must be NULL (MOE_ERR_INVALID_ARG otherwise).
 * logits (device): [T, E] fp32. out (device): [T, H] bf16.
 * ws (device): at least moe_workspace_size bytes. */
MOE_API moe_status_t moe_layer_forward(moe_handle_t h, const moe_config_t* cfg,
                                       const moe_weights_t* w, const void* x,
                                       const uint8_t* x_scale_or_null, const float* logits,
                                       void* out, void* ws, size_t ws_bytes, moe_stream_t main,
                                       moe_stream_t side);

/* Gating + routing ([Hy3] section 8.5: the main stream runs gating, then the
 * routed path): logits = x w_router^T in fp32 (bf16 inputs), then the
 * routing of moe_route. With E <= 256 one kernel does both. Up to 256
 * tokens it is a CUDA-core split-K kernel (a cluster of 8 CTAs per group of
 * tokens, partial sums added in a fixed order, top-k by one warp per token);
 * above that a tensor-core GEMM with the top-k in its epilogue on the fp32
 * accumulators. Either way the result does not depend on logits_out.
 * x (device): [T, H] bf16; w_router (device): [E, H] bf16;
 * logits_out (device, nullable when E <= 256): [T, E] fp32;
 * topk_idx / topk_w (device): [T, K]. E > 256 needs E % 32 == 0. */
MOE_API moe_status_t moe_gate_route(moe_handle_t h, const moe_config_t* cfg, const void* x,
                                    const void* w_router, float* logits_out, int32_t* topk_idx,
                                    float* topk_w, moe_stream_t stream);

/* moe_layer_forward with the gating projection inside: routes from
 * x w_router^T (moe_gate_route) instead of given logits. In MXFP8 mode the
 * router reads the bf16 x. E > 256 needs E % 32 == 0. */
MOE_API moe_status_t moe_layer_forward_gated(moe_handle_t h, const moe_config_t* cfg,
                                             const moe_weights_t* w, const void* w_router,
                                             const void* x, void* out, void* ws, size_t ws_bytes,
                                             moe_stream_t main, moe_stream_t side);

/* The same layer with HOST activations: copies x_host [T, H] bf16 and
 * logits_host [T, E] fp32 to the device (staging inside ws), runs
 * moe_layer_forward, copies out back to out_host [T, H] bf16 and
 * synchronises `main`. Weights stay device-resident. Host buffers should be
 * pinned for asynchronous copies. */
MOE_API moe_status_t moe_layer_forward_host(moe_handle_t h, const moe_config_t* cfg,
                                            const moe_weights_t* w, const void* x_host,
                                            const float* logits_host, void* out_host, void* ws,
                                            size_t ws_bytes, moe_stream_t main, moe_stream_t side);

/* Read and clear the handle's device status word (synchronises `stream`).
 * *code = 0 when no device-side error was recorded since the last read;
 * otherwise the code of the first failure (see the MOE_DEV_* values below)
 * and the call returns MOE_ERR_DEVICE_TIMEOUT for wait timeouts or
 * MOE_ERR_INVALID_ARG for bad expert ids / permutation indices. */
MOE_API moe_status_t moe_get_device_status(moe_handle_t h, int* code, moe_stream_t stream);

enum {
  MOE_DEV_OK = 0,
  MOE_DEV_TIMEOUT_PRODUCER = 1, /* GEMM TMA producer gave up waiting */
  MOE_DEV_TIMEOUT_MMA = 2,      /* GEMM MMA issuer gave up waiting */
  MOE_DEV_TIMEOUT_EPILOGUE = 3, /* GEMM epilogue gave up waiting */
  MOE_DEV_TIMEOUT_SELFTEST = 4, /* moe_selftest_wait_timeout's wait */
  MOE_DEV_BAD_EXPERT_ID = 16,   /* moe_permute saw an id outside [0, E) */
  MOE_DEV_BAD_PERM_INDEX = 17   /* a permutation index out of range */
};

/* Average device time per stage (ms) over the last calls of
 * moe_layer_forward made with MOE_OPT_STAGE_TIMING on (at most 512; the
 * window restarts after each read). ms: MOE_NUM_STAGES floats out (-1 for a
 * stage that did not run). *n_calls: calls averaged. Synchronises the
 * recorded events. */
MOE_API moe_status_t moe_read_stage_times(moe_handle_t h, float* ms, int* n_calls);

/* Permutation with no workspace and no allocation (the paper has no
 * counterpart; this exists for callers of this library that cannot call
 * cudaMalloc and have no workspace to hand over, such as a plugin inside an
 * engine that owns every device allocation, or code that must not allocate
 * after start-up).
 * Same arguments, results and kernels as moe_permute, minus ws/ws_bytes. Up
 * to 262144 (token, slot) pairs the permutation needs no scratch at all;
 * above that the per-warp histogram lives in a fixed array in the library's
 * own device memory, MOE_PERMUTE_STATIC_MAX_HIST_INTS int32 (1 MiB), which
 * every GPU that loads the library holds until the process exits.
 * Limit: E * ceil(T*K / 256) <= MOE_PERMUTE_STATIC_MAX_HIST_INTS (for E = 192
 * and K = 8: T <= 43690); larger sizes return MOE_ERR_WORKSPACE before any
 * launch.
 * MXFP8 and W4A8 configs move the 1-byte E4M3 rows of x and their E8M0
 * scales exactly as moe_permute does (same H rule: H % 128 == 0).
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it for the life of the process; make that first
 * call before any stream capture. The cache does not survive cudaDeviceReset:
 * do not call this entry point on a device after resetting it. The caller's
 * current device is restored before the call returns. The call never
 * allocates or frees device memory.
 * All calls on a device share the one array and each call overwrites it:
 * calls that overlap on the GPU (different streams, no ordering between
 * them) race and give undefined results. Nothing in the array needs to
 * start at zero. */
#define MOE_PERMUTE_STATIC_MAX_HIST_INTS 262144
MOE_API moe_status_t moe_permute_static_scratch(moe_handle_t h, const moe_config_t* cfg,
                                                const void* x, const uint8_t* x_scale,
                                                const int32_t* topk_idx, int32_t* counts,
                                                int32_t* offsets, int32_t* perm_src,
                                                int32_t* flat_to_perm, void* x_perm,
                                                uint8_t* x_perm_scale, moe_stream_t stream);

/* Launch one block whose thread waits on an mbarrier that nothing ever
 * arrives on, with the handle's wait limit; the wait gives up, records
 * MOE_DEV_TIMEOUT_SELFTEST in the status word and the kernel returns. Used to
 * test the bounded-wait path without hanging the GPU. */
MOE_API moe_status_t moe_selftest_wait_timeout(moe_handle_t h, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
