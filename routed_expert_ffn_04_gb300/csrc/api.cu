// C-ABI entry points: argument validation, the handle (device, SM count,
// status word, events), workspace carving, and the two-stream orchestration
// of the whole layer.
//
// Orchestration follows "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战",
// section 8.5 (the shared expert depends only on the MoE input, runs on a
// second stream whose start is synchronised after gating, and is hidden under
// the routed path) and "HunyuanImage-3.0 MoE 多流变体实战", 源码级实现拆解 §1-§3
// (a side stream handed in at construction; an input-ready event recorded on
// the main stream and waited on by the side stream; an mlp-done event
// recorded on the side stream and waited on by the main stream before
// output = hidden_states_mlp + combined_output). Gating (the logits) is an
// input here, so the side stream may start at entry.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/moe.h"
#include "internal.h"

using namespace moe;

namespace {

constexpr int kTimingRing = 512;
constexpr int kEventsPerCall = 9;  // main: 0 entry,1 route,2 permute,3 g1,4 g2,5 combine; side: 6 start,7 end; 8 spare

}  // namespace

struct moe_handle {
  int device = 0;
  int num_sms = 0;
  int* status = nullptr;  // device word (64 bytes allocated)
  cudaEvent_t ev_in = nullptr, ev_sh = nullptr;
  int gemm_mode = kModeAuto;
  int stage_timing = 0;
  int shared_fold = 0;  // MOE_OPT_SHARED_FOLD
  int shared_sms = 0;   // MOE_OPT_SHARED_SMS: 0 no split, k > 0 fixed
  int gather_a = 1;     // MOE_OPT_GATHER_A
  int mx_tile = 0;      // MOE_OPT_MX_TILE
  uint64_t wait_limit_ns = kDefaultWaitLimitNs;
  cudaEvent_t* tev = nullptr;  // [kTimingRing][kEventsPerCall], created on first use
  int t_calls = 0;             // calls recorded since the last read
  bool t_shared[kTimingRing] = {};
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__global__ void set_i32_kernel(int32_t* p, int v) { *p = v; }

bool is_mx(int dtype) { return dtype == MOE_MXFP8_E4M3 || dtype == MOE_MXFP4_W4A8; }

// Packed E2M1 weights are read through tensor maps that need 32-byte bases.
bool weights_aligned32(const void* a, const void* b, const void* c) {
  return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
           reinterpret_cast<uintptr_t>(c)) & 31) == 0;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_cfg(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H <= 0 || c->E <= 0 || c->K <= 0 || c->I <= 0 || c->I_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->K > c->E || c->K > 32 || c->E > 1024) return MOE_ERR_INVALID_ARG;
  if (c->H % 64 || c->I % 64 || c->I_shared % 64) return MOE_ERR_INVALID_ARG;
  if ((long long)c->T * c->K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  const long long wide = c->H > c->I ? c->H : c->I;
  if ((long long)c->T * c->K * wide >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_BF16 && !is_mx(c->dtype)) return MOE_ERR_INVALID_ARG;
  // MX: whole scale atoms (128 x 128) along H, I and I_shared.
  if (is_mx(c->dtype) && (c->H % 128 || c->I % 128 || c->I_shared % 128))
    return MOE_ERR_INVALID_ARG;
  if (!(c->scaling == c->scaling)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// The shared expert can run as one more group of the routed grouped GEMM
// (MOE_OPT_SHARED_FOLD): bf16, the same intermediate size, a group to spare.
bool foldable(const moe_config_t* c) {
  return c->dtype == MOE_BF16 && c->I_shared > 0 && c->I_shared == c->I && c->E + 1 <= 1024;
}

// SMs the shared expert gets while it runs beside the routed path on the side
// stream (0: no split, the default). Measured on the decode, MX, skewed and
// prefill workloads, no fixed split beat letting both streams' persistent
// grids take every SM: the shared kernels then fill the SMs that the short
// routing and permutation stages leave idle.
int shared_sm_budget(int num_sms, int option) {
  if (option <= 0 || num_sms < 4) return 0;
  const int cap = num_sms / 2;
  return option < cap ? option : cap;
}

// Workspace layout of moe_layer_forward, every piece 256-byte aligned.
struct Layout {
  size_t topk_idx, topk_w, counts, offsets, tile_offsets, perm_src, flat_to_perm, perm_scratch, x_perm, h,
      y_perm, s, h_shared, x_stage, logits_stage, out_stage, x_mx, total;
  // MXFP8 only: E8M0 scales of x (x_mx holds its E4M3 codes) row-major and
  // as scale atoms; atoms of the permuted x, of h and of the shared expert's h.
  size_t x_mx_s, x_mx_atoms, x_perm_s, h_s, h_shared_s;
};

Layout layout_of(const moe_config_t* c) {
  Layout L;
  const size_t T = c->T, H = c->H, E = c->E, K = c->K, I = c->I, Is = c->I_shared, TK = T * K;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return at;
  };
  L.topk_idx = take(TK * 4);
  L.topk_w = take(TK * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 2) * 4);  // + the folded shared group's end
  L.tile_offsets = take((E + 1) * 4);
  L.perm_src = take(TK * 4);
  L.flat_to_perm = take(TK * 4);
  L.perm_scratch = take(permute_scratch_bytes((int)TK, (int)E));
  const bool mx = is_mx(c->dtype);
  const size_t eb = mx ? 1 : 2;  // bytes per activation element (E4M3 codes or bf16)
  // Foldable layers keep room for the shared expert's T rows after the routed ones.
  const size_t RX = TK + (foldable(c) ? T : 0);
  L.x_perm = take(RX * H * eb);
  L.h = take(RX * I * eb);
  L.y_perm = take(RX * H * 4);
  L.s = take(Is ? T * H * 4 : 0);
  L.h_shared = take(T * Is * eb);
  L.x_stage = take(T * H * 2);
  L.logits_stage = take(T * E * 4);
  L.out_stage = take(T * H * 2);
  L.x_mx = take(mx ? T * H : 0);
  L.x_mx_s = take(mx ? T * H / 32 : 0);
  L.x_mx_atoms = take(mx ? scale_atom_bytes(T, 1, (int)H) : 0);
  L.x_perm_s = take(mx ? scale_atom_bytes(TK, (int)E, (int)H) : 0);
  L.h_s = take(mx ? scale_atom_bytes(TK, (int)E, (int)I) : 0);
  L.h_shared_s = take(mx ? scale_atom_bytes(T, 1, (int)Is) : 0);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

moe_status_t check_handle(moe_handle_t h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ERR_CUDA;
  if (cur != h->device && cudaSetDevice(h->device) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

GroupedGemmArgs gemm_args(moe_handle_t h, int G, const int32_t* offsets, int rows, int H, int I,
                          const void* a, const void* wg, const void* wu, const void* wd, void* hbuf,
                          float* y, const uint8_t* sg = nullptr, const uint8_t* sd = nullptr) {
  GroupedGemmArgs g;
  g.a_scale = nullptr;
  g.h_scale = nullptr;
  g.topk_idx = nullptr;
  g.topk_w = nullptr;
  g.topk = 0;
  g.scaling = 1.0f;
  g.route_norm = 0;
  g.s_gate = sg;
  g.s_down = sd;
  g.w4 = 0;
  g.mx_tile = 0;
  g.shared_w_gate = nullptr;
  g.shared_w_up = nullptr;
  g.shared_w_down = nullptr;
  g.gather_src = nullptr;
  g.gather_k = 0;
  g.gather_x = nullptr;
  g.G = G;
  g.offsets = offsets;
  g.rows = rows;
  g.H = H;
  g.I = I;
  g.a = a;
  g.w_gate = wg;
  g.w_up = wu;
  g.w_down = wd;
  g.h = hbuf;
  g.y = y;
  g.mode = h->gemm_mode;
  g.mx_tile = h->mx_tile;
  g.num_sms = h->num_sms;
  g.status = h->status;
  g.wait_limit_ns = h->wait_limit_ns;
  return g;
}

cudaError_t timing_events(moe_handle_t h) {
  if (h->tev) return cudaSuccess;
  h->tev = new (std::nothrow) cudaEvent_t[kTimingRing * kEventsPerCall];
  if (!h->tev) return cudaErrorMemoryAllocation;
  for (int i = 0; i < kTimingRing * kEventsPerCall; ++i) {
    cudaError_t e = cudaEventCreate(&h->tev[i]);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Gating ([Hy3] section 8.5: the main stream runs gating, then the routed
// path): logits = x W_router^T and the routing of step 1. E <= 256 runs as
// one kernel with the top-k in the GEMM epilogue; larger E writes the logits
// (into `logits`, required then) and runs the routing kernel on them.
cudaError_t gate_route(moe_handle_t h, const moe_config_t* c, const void* x, const void* w_router,
                       float* logits, int32_t* topk_idx, float* topk_w, cudaStream_t s) {
  if (gate_route_small_fits(c->T, c->H, c->E))
    return launch_gate_route_small(x, w_router, c->T, c->H, c->E, c->K, c->scaling, c->route_norm,
                                   logits, topk_idx, topk_w, s);
  GroupedGemmArgs g = gemm_args(h, 1, nullptr, c->T, /*H (N)=*/c->E, /*I (K)=*/c->H, x, nullptr,
                                nullptr, w_router, const_cast<void*>(x), logits);
  if (c->E <= 256) {
    g.topk_idx = topk_idx;
    g.topk_w = topk_w;
    g.topk = c->K;
    g.scaling = c->scaling;
    g.route_norm = c->route_norm;
    return launch_gate_route(g, s);
  }
  cudaError_t e = launch_gemm_down(g, s);
  if (e == cudaSuccess)
    e = launch_route(logits, c->T, c->E, c->K, c->scaling, c->route_norm, topk_idx, topk_w, s);
  return e;
}

}  // namespace

namespace moe {
int handle_device(moe_handle_t h) { return h->device; }
int* handle_status_word(moe_handle_t h) { return h->status; }
}  // namespace moe

extern "C" {

MOE_API const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

MOE_API moe_status_t moe_create(int device, moe_handle_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major < 10) return MOE_ERR_UNSUPPORTED;
  if (!gemm_init_driver()) return MOE_ERR_CUDA;
  moe_handle* h = new (std::nothrow) moe_handle();
  if (!h) return MOE_ERR_CUDA;
  h->device = device;
  h->num_sms = sms;
  if (gemm_prepare_device() != cudaSuccess || gemm_mx_prepare_device() != cudaSuccess ||
      permute_prepare_device() != cudaSuccess ||
      gate_small_prepare_device() != cudaSuccess ||
      cudaMalloc(&h->status, 64) != cudaSuccess ||
      cudaMemset(h->status, 0, 64) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&h->ev_sh, cudaEventDisableTiming) != cudaSuccess) {
    moe_destroy(h);
    return MOE_ERR_CUDA;
  }
  *out = h;
  return MOE_OK;
}

MOE_API moe_status_t moe_destroy(moe_handle_t h) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaSetDevice(h->device);
  if (h->status) cudaFree(h->status);
  if (h->ev_in) cudaEventDestroy(h->ev_in);
  if (h->ev_sh) cudaEventDestroy(h->ev_sh);
  if (h->tev) {
    for (int i = 0; i < kTimingRing * kEventsPerCall; ++i)
      if (h->tev[i]) cudaEventDestroy(h->tev[i]);
    delete[] h->tev;
  }
  delete h;
  return MOE_OK;
}

MOE_API moe_status_t moe_set_option(moe_handle_t h, moe_option_t opt, int value) {
  if (!h) return MOE_ERR_INVALID_ARG;
  switch (opt) {
    case MOE_OPT_GEMM_MODE:
      if (value < 0 || value > 3) return MOE_ERR_INVALID_ARG;
      h->gemm_mode = value;
      return MOE_OK;
    case MOE_OPT_STAGE_TIMING:
      h->stage_timing = value ? 1 : 0;
      h->t_calls = 0;
      return MOE_OK;
    case MOE_OPT_WAIT_LIMIT_US:
      if (value <= 0) return MOE_ERR_INVALID_ARG;
      h->wait_limit_ns = (uint64_t)value * 1000ull;
      return MOE_OK;
    case MOE_OPT_SHARED_FOLD:
      h->shared_fold = value ? 1 : 0;
      return MOE_OK;
    case MOE_OPT_SHARED_SMS:
      if (value < 0) return MOE_ERR_INVALID_ARG;
      h->shared_sms = value;
      return MOE_OK;
    case MOE_OPT_GATHER_A:
      h->gather_a = value ? 1 : 0;
      return MOE_OK;
    case MOE_OPT_MX_TILE:
      if (value < 0 || value > 3) return MOE_ERR_INVALID_ARG;
      h->mx_tile = value;
      return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

MOE_API moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  *bytes = layout_of(cfg).total;
  return MOE_OK;
}

MOE_API moe_status_t moe_route(moe_handle_t h, const moe_config_t* cfg, const float* logits,
                               int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!logits || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w)) return MOE_ERR_INVALID_ARG;
  if ((st = check_handle(h)) != MOE_OK) return st;
  return cuda_status(launch_route(logits, cfg->T, cfg->E, cfg->K, cfg->scaling, cfg->route_norm,
                                  topk_idx, topk_w, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_permute_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  *bytes = permute_scratch_bytes(cfg->T * cfg->K, cfg->E);
  return MOE_OK;
}

MOE_API moe_status_t moe_permute(moe_handle_t h, const moe_config_t* cfg, const void* x,
                                 const uint8_t* x_scale, const int32_t* topk_idx, int32_t* counts,
                                 int32_t* offsets, int32_t* perm_src, int32_t* flat_to_perm,
                                 void* x_perm, uint8_t* x_perm_scale, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  const bool mx = is_mx(cfg->dtype);
  const bool any = cfg->T > 0;
  if (!counts || !offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (any && (!x || !topk_idx || !perm_src || !flat_to_perm || !x_perm)) return MOE_ERR_INVALID_ARG;
  if (any && mx && (!x_scale || !x_perm_scale)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, topk_idx, counts, offsets, perm_src, flat_to_perm, x_perm, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (mx && (!aligned16(x_scale) || !aligned16(x_perm_scale))) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < permute_scratch_bytes(cfg->T * cfg->K, cfg->E)) return MOE_ERR_WORKSPACE;
  if ((st = check_handle(h)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int TK = cfg->T * cfg->K;
  cudaError_t e = launch_permute_index(topk_idx, TK, cfg->E, ws, counts, offsets, nullptr,
                                       perm_src, flat_to_perm, h->status, s);
  if (e == cudaSuccess)
    e = launch_scatter_rows(x, cfg->T, mx ? cfg->H : cfg->H * 2, flat_to_perm, cfg->K, TK, x_perm,
                            h->status, s);
  if (e == cudaSuccess && mx)
    e = launch_scatter_rows(x_scale, cfg->T, cfg->H / 32, flat_to_perm, cfg->K, TK, x_perm_scale,
                            h->status, s);
  return cuda_status(e);
}

namespace {
// moe_grouped_swiglu_gemm workspace: h, then (MXFP8) the scale atoms of h and of a.
struct GemmWs {
  size_t h, h_atoms, a_atoms, total;
};
GemmWs gemm_ws(int rows, int groups, int H, int I, bool mx) {
  GemmWs L;
  L.h = 0;
  L.h_atoms = align_up((size_t)rows * I * (mx ? 1 : 2) + 1, 256);
  L.a_atoms = L.h_atoms + (mx ? align_up(scale_atom_bytes(rows, groups, I) + 1, 256) : 0);
  L.total = L.a_atoms + (mx ? align_up(scale_atom_bytes(rows, groups, H) + 1, 256) : 0);
  return L;
}
}  // namespace

MOE_API moe_status_t moe_grouped_gemm_workspace_size(int rows, int num_groups, int H, int I,
                                                     moe_dtype_t dtype, size_t* bytes) {
  if (!bytes || rows < 0 || num_groups <= 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && !is_mx(dtype)) return MOE_ERR_INVALID_ARG;
  *bytes = gemm_ws(rows, num_groups, H, I, is_mx(dtype)).total;
  return MOE_OK;
}

MOE_API moe_status_t moe_grouped_swiglu_gemm(moe_handle_t h, int num_groups, int rows, int H,
                                             int I, moe_dtype_t dtype, const void* a,
                                             const uint8_t* a_scale, const int32_t* offsets,
                                             const void* w_gate, const void* w_up,
                                             const void* w_down, const uint8_t* s_gate,
                                             const uint8_t* s_up, const uint8_t* s_down, float* y,
                                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (num_groups <= 0 || num_groups > 1024 || rows < 0 || H <= 0 || I <= 0 || H % 64 || I % 64)
    return MOE_ERR_INVALID_ARG;
  if (offsets == nullptr && num_groups != 1) return MOE_ERR_INVALID_ARG;
  if ((long long)rows * (H > I ? H : I) >= (1ll << 40)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_BF16 && !is_mx(dtype)) return MOE_ERR_INVALID_ARG;
  const bool mx = is_mx(dtype);
  const bool w4 = dtype == MOE_MXFP4_W4A8;
  // W4A8: w_gate holds the gate and up codes together, w_up is unused.
  if (!a || !w_gate || (!w_up && !w4) || !w_down || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (mx && (!a_scale || !s_gate || !s_down || H % 128 || I % 128)) return MOE_ERR_INVALID_ARG;
  if (w4 && !weights_aligned32(w_gate, w_up, w_down)) return MOE_ERR_INVALID_ARG;
  (void)s_up;  // MXFP8: s_gate holds the gate and up scale atoms together
  const void* ptrs[] = {a, offsets, w_gate, w_up, w_down, y, ws, s_gate, s_down};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  const GemmWs W = gemm_ws(rows, num_groups, H, I, mx);
  if (ws_bytes < W.total) return MOE_ERR_WORKSPACE;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GroupedGemmArgs g = gemm_args(h, num_groups, offsets, rows, H, I, a, w_gate, w_up, w_down, ws, y,
                                mx ? s_gate : nullptr, mx ? s_down : nullptr);
  g.w4 = w4;
  cudaError_t e = cudaSuccess;
  if (mx) {  // block-scaled tensor cores; h stays E4M3 + E8M0 between the GEMMs
    uint8_t* a_atoms = at<uint8_t>(ws, W.a_atoms);
    e = launch_gather_scale_atoms(a_scale, rows, H, nullptr, 1, offsets, num_groups, rows, a_atoms,
                                  h->status, s);
    g.a_scale = a_atoms;
    g.h_scale = at<uint8_t>(ws, W.h_atoms);
    if (e == cudaSuccess) e = launch_gemm_mx_gate_up(g, s);
    if (e == cudaSuccess) e = launch_gemm_mx_down(g, s);
  } else {
    e = launch_gemm_gate_up(g, s);
    if (e == cudaSuccess) e = launch_gemm_down(g, s);
  }
  return cuda_status(e);
}

MOE_API moe_status_t moe_combine(moe_handle_t h, const moe_config_t* cfg, const float* y_perm,
                                 const float* topk_w, const int32_t* flat_to_perm,
                                 const float* shared_out, void* out, moe_stream_t stream) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!y_perm || !topk_w || !flat_to_perm || !out)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {y_perm, topk_w, flat_to_perm, shared_out, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if ((st = check_handle(h)) != MOE_OK) return st;
  return cuda_status(launch_combine(y_perm, topk_w, flat_to_perm, shared_out, cfg->T, cfg->K,
                                    cfg->H, out, h->status, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_pack_mx_scales(moe_handle_t h, const uint8_t* scale0,
                                        const uint8_t* scale1, int64_t rows, int cols,
                                        uint8_t* atoms, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 128) return MOE_ERR_INVALID_ARG;
  if (rows % (scale1 ? 64 : 128)) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!scale0 || !atoms)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(scale0) || !aligned16(scale1) || !aligned16(atoms)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  return cuda_status(
      launch_pack_weight_scales(scale0, scale1, rows, cols, atoms, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_tile_mxfp4_weights(moe_handle_t h, const uint8_t* q0, const uint8_t* q1, int64_t rows,
                                            int cols, uint8_t* tiled, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 128 || rows % 128) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!q0 || !tiled || q0 == tiled || q1 == tiled)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(q0) || !aligned16(q1) || !aligned16(tiled)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  return cuda_status(launch_tile_e2m1(q0, q1, rows, cols, tiled, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_quantize_mxfp4(moe_handle_t h, const void* in_bf16, int64_t rows,
                                        int cols, uint8_t* q, uint8_t* scale, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 32) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!in_bf16 || !q || !scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(in_bf16) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  return cuda_status(launch_mx4_quantize(in_bf16, rows, cols, q, scale, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_quantize_mxfp8(moe_handle_t h, const void* in_bf16, int64_t rows,
                                        int cols, uint8_t* q, uint8_t* scale, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 32) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!in_bf16 || !q || !scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(in_bf16) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  return cuda_status(
      launch_mx_quantize(in_bf16, rows, cols, q, scale, nullptr,
                         static_cast<cudaStream_t>(stream)));
}

static moe_status_t layer_forward_impl(moe_handle_t h, const moe_config_t* cfg,
                                       const moe_weights_t* w, const void* x,
                                       const uint8_t* x_scale, const float* logits,
                                       const void* w_router, void* out, void* ws, size_t ws_bytes,
                                       moe_stream_t main, moe_stream_t side) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!w || !ws) return MOE_ERR_INVALID_ARG;
  const bool has_shared = cfg->I_shared > 0;
  if (cfg->T > 0 && (!x || (!logits && !w_router) || !out)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  const bool mx = is_mx(cfg->dtype);
  const bool w4 = cfg->dtype == MOE_MXFP4_W4A8;  // routed experts E2M1; shared stays E4M3
  // W4A8: w_gate holds the routed gate and up codes together, w_up is unused.
  if (!w->w_gate || (!w->w_up && !w4) || !w->w_down) return MOE_ERR_INVALID_ARG;
  if (has_shared && (!w->ws_gate || !w->ws_up || !w->ws_down)) return MOE_ERR_INVALID_ARG;
  // Pre-quantised activations: only in MX mode, and only with given logits
  // (the router reads bf16 x).
  if (x_scale && (!mx || w_router)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_scale)) return MOE_ERR_INVALID_ARG;
  if (mx && (!w->s_gate || !w->s_down)) return MOE_ERR_INVALID_ARG;
  if (w4 && !weights_aligned32(w->w_gate, w->w_up, w->w_down)) return MOE_ERR_INVALID_ARG;
  if (mx && has_shared && (!w->ss_gate || !w->ss_down)) return MOE_ERR_INVALID_ARG;
  if (mx && (!aligned16(w->s_gate) || !aligned16(w->s_down) || !aligned16(w->ss_gate) ||
             !aligned16(w->ss_down)))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, logits, out, ws, w->w_gate, w->w_up, w->w_down, w->ws_gate, w->ws_up, w->ws_down};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(cfg);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if ((st = check_handle(h)) != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;

  cudaStream_t sm = static_cast<cudaStream_t>(main);
  cudaStream_t ss = static_cast<cudaStream_t>(side);
  const int T = cfg->T, H = cfg->H, E = cfg->E, K = cfg->K, I = cfg->I, Is = cfg->I_shared;
  const int TK = T * K;
  int32_t* topk_idx = at<int32_t>(ws, L.topk_idx);
  float* topk_w = at<float>(ws, L.topk_w);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* perm_src = at<int32_t>(ws, L.perm_src);
  int32_t* flat_to_perm = at<int32_t>(ws, L.flat_to_perm);
  void* x_perm = at<void>(ws, L.x_perm);
  void* hbuf = at<void>(ws, L.h);
  float* y_perm = at<float>(ws, L.y_perm);
  float* s_out = has_shared ? at<float>(ws, L.s) : nullptr;
  void* h_shared = at<void>(ws, L.h_shared);

  // Stage timing: events on the main stream between stages (and on the side stream).
  cudaEvent_t* ev = nullptr;
  int slot = 0;
  if (h->stage_timing) {
    if (timing_events(h) != cudaSuccess) return MOE_ERR_CUDA;
    slot = h->t_calls % kTimingRing;
    ev = h->tev + slot * kEventsPerCall;
    h->t_shared[slot] = has_shared && !(h->shared_fold && foldable(cfg));
  }
  auto mark = [&](int i, cudaStream_t s) {
    if (ev) cudaEventRecord(ev[i], s);
  };

  cudaError_t e = cudaSuccess;
  mark(0, sm);
  const void* x_gate = x;  // the router reads x as given (bf16)
  const uint8_t* xq_s = nullptr;  // MX: row-major E8M0 scales of the E4M3 x
  if (mx && x_scale) {
    // The caller's E4M3 codes and scales; the shared expert still needs its
    // scales as atoms (one group of T rows).
    xq_s = x_scale;
    if (has_shared)
      e = launch_gather_scale_atoms(x_scale, T, H, nullptr, 1, nullptr, 1, T,
                                    at<uint8_t>(ws, L.x_mx_atoms), h->status, sm);
  } else if (mx) {  // dynamic MXFP8 quantisation of x (E4M3 codes + E8M0 scales)
    void* xq = at<void>(ws, L.x_mx);
    uint8_t* s = at<uint8_t>(ws, L.x_mx_s);
    e = launch_mx_quantize(x, T, H, static_cast<uint8_t*>(xq), s,
                           has_shared ? at<uint8_t>(ws, L.x_mx_atoms) : nullptr, sm);
    xq_s = s;
    x = xq;
  }
  cudaStream_t s_sh = ss ? ss : sm;
  // Gated: the gating projection and the routing run first, and the side
  // stream forks after them ([Hy3] section 8.5: gating, then the shared
  // expert beside the routed path), so the gating kernel does not queue
  // behind the shared expert's persistent GEMMs for SMs.
  if (e == cudaSuccess && w_router) {
    e = gate_route(h, cfg, x_gate, w_router, at<float>(ws, L.logits_stage), topk_idx, topk_w, sm);
    mark(1, sm);
  }
  // Folded: the shared expert is group E of the routed GEMMs (rows TK..TK+T-1
  // of x_perm, h and y_perm), so nothing runs on the side stream.
  const bool fold = h->shared_fold && foldable(cfg);
  // Optionally the shared expert's GEMMs get a few SMs of their own and the
  // routed GEMMs the rest (MOE_OPT_SHARED_SMS; off by default).
  const int k_sh = (has_shared && !fold && ss) ? shared_sm_budget(h->num_sms, h->shared_sms) : 0;
  if (has_shared && !fold) {
    if (ss) {
      e = cudaEventRecord(h->ev_in, sm);  // input ready on main
      if (e == cudaSuccess) e = cudaStreamWaitEvent(ss, h->ev_in, 0);
    }
    mark(6, s_sh);
    GroupedGemmArgs g = gemm_args(h, 1, nullptr, T, H, Is, x, w->ws_gate, w->ws_up, w->ws_down,
                                  h_shared, s_out, mx ? w->ss_gate : nullptr,
                                  mx ? w->ss_down : nullptr);
    // Beside the routed path the shared MLP should finish early rather than
    // use few SMs well: up to 128 tokens its weights fill the MMA rows
    // (more CTAs stream them) unless a tiling is forced.
    if (!mx && g.mode == kModeAuto && T <= 128) g.mode = kModeWeightsM;
    if (k_sh > 0) g.num_sms = k_sh;
    if (mx) {
      g.a_scale = at<uint8_t>(ws, L.x_mx_atoms);
      g.h_scale = at<uint8_t>(ws, L.h_shared_s);
      if (e == cudaSuccess) e = launch_gemm_mx_gate_up(g, s_sh);
      if (e == cudaSuccess) e = launch_gemm_mx_down(g, s_sh);
    } else {
      if (e == cudaSuccess) e = launch_gemm_gate_up(g, s_sh);
      if (e == cudaSuccess) e = launch_gemm_down(g, s_sh);
    }
    mark(7, s_sh);
    if (e == cudaSuccess && ss) e = cudaEventRecord(h->ev_sh, ss);  // shared MLP done
  }
  if (!w_router) {
    if (e == cudaSuccess)
      e = launch_route(logits, T, E, K, cfg->scaling, cfg->route_norm, topk_idx, topk_w, sm);
    mark(1, sm);
  }
  int32_t* tile_offsets = mx ? at<int32_t>(ws, L.tile_offsets) : nullptr;
  if (e == cudaSuccess)
    e = launch_permute_index(topk_idx, TK, E, at<void>(ws, L.perm_scratch), counts, offsets,
                             tile_offsets, perm_src, flat_to_perm, h->status, sm);
  GroupedGemmArgs g = gemm_args(h, fold ? E + 1 : E, offsets, fold ? TK + T : TK, H, I, x_perm,
                                w->w_gate, w->w_up, w->w_down, hbuf, y_perm,
                                mx ? w->s_gate : nullptr, mx ? w->s_down : nullptr);
  g.w4 = w4;
  if (k_sh > 0) g.num_sms = h->num_sms - k_sh;
  if (fold) {
    g.shared_w_gate = w->ws_gate;
    g.shared_w_up = w->ws_up;
    g.shared_w_down = w->ws_down;
  }
  if (mx) {
    g.a_scale = at<uint8_t>(ws, L.x_perm_s);
    g.h_scale = at<uint8_t>(ws, L.h_s);
  }
  // bf16, tokens-as-M: GEMM-1 gathers its A rows from x itself (InitRouting's
  // row gather fused into the grouped GMM's load), so x_perm is not written.
  const bool gather = !mx && !fold && h->gather_a && gemm_pick_mode(g) == kModeTokensM;
  if (gather) {
    g.gather_src = perm_src;
    g.gather_k = K;
    g.gather_x = x;
  }
  // MX: the E4M3 rows and their scale atoms in one pass; bf16: the rows.
  if (e == cudaSuccess && !gather)
    e = mx ? launch_scatter_rows_mx(static_cast<const uint8_t*>(x), xq_s, T, H, flat_to_perm,
                                    topk_idx, offsets, tile_offsets, K, TK, E,
                                    static_cast<uint8_t*>(x_perm), at<uint8_t>(ws, L.x_perm_s),
                                    h->status, sm)
           : launch_scatter_rows(x, T, H * 2, flat_to_perm, K, TK, x_perm, h->status, sm);
  if (e == cudaSuccess && fold) {  // group E: x itself, after the routed rows
    set_i32_kernel<<<1, 1, 0, sm>>>(offsets + E + 1, TK + T);
    e = cudaGetLastError();
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(x_perm) + (size_t)TK * H * 2, x, (size_t)T * H * 2,
                          cudaMemcpyDeviceToDevice, sm);
  }
  mark(2, sm);
  if (e == cudaSuccess) e = mx ? launch_gemm_mx_gate_up(g, sm) : launch_gemm_gate_up(g, sm);
  mark(3, sm);
  if (e == cudaSuccess) e = mx ? launch_gemm_mx_down(g, sm) : launch_gemm_down(g, sm);
  mark(4, sm);
  if (e == cudaSuccess && has_shared && ss && !fold) e = cudaStreamWaitEvent(sm, h->ev_sh, 0);
  if (e == cudaSuccess)
    e = launch_combine(y_perm, topk_w, flat_to_perm, fold ? y_perm + (size_t)TK * H : s_out, T, K, H,
                       out, h->status, sm);
  mark(5, sm);
  if (ev) h->t_calls += 1;
  return cuda_status(e);
}

MOE_API moe_status_t moe_layer_forward(moe_handle_t h, const moe_config_t* cfg,
                                       const moe_weights_t* w, const void* x,
                                       const uint8_t* x_scale_or_null, const float* logits,
                                       void* out, void* ws, size_t ws_bytes, moe_stream_t main,
                                       moe_stream_t side) {
  if (cfg && cfg->T > 0 && !logits) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(h, cfg, w, x, x_scale_or_null, logits, nullptr, out, ws, ws_bytes,
                            main, side);
}

MOE_API moe_status_t moe_layer_forward_gated(moe_handle_t h, const moe_config_t* cfg,
                                             const moe_weights_t* w, const void* w_router,
                                             const void* x, void* out, void* ws, size_t ws_bytes,
                                             moe_stream_t main, moe_stream_t side) {
  if (!w_router || (cfg && cfg->E > 256 && cfg->E % 32)) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(h, cfg, w, x, nullptr, nullptr, w_router, out, ws, ws_bytes, main,
                            side);
}

MOE_API moe_status_t moe_gate_route(moe_handle_t h, const moe_config_t* cfg, const void* x,
                                    const void* w_router, float* logits_out, int32_t* topk_idx,
                                    float* topk_w, moe_stream_t stream) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!x || !w_router || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (cfg->E > 256 && cfg->T > 0 && !logits_out) return MOE_ERR_INVALID_ARG;
  if (cfg->E > 256 && cfg->E % 32) return MOE_ERR_INVALID_ARG;  // logits GEMM stores 32-column chunks
  const void* ptrs[] = {x, w_router, logits_out, topk_idx, topk_w};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if ((st = check_handle(h)) != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  return cuda_status(gate_route(h, cfg, x, w_router, logits_out, topk_idx, topk_w,
                                static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status_t moe_layer_forward_host(moe_handle_t h, const moe_config_t* cfg,
                                            const moe_weights_t* w, const void* x_host,
                                            const float* logits_host, void* out_host, void* ws,
                                            size_t ws_bytes, moe_stream_t main, moe_stream_t side) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!ws || (cfg->T > 0 && (!x_host || !logits_host || !out_host))) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(cfg);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if ((st = check_handle(h)) != MOE_OK) return st;
  cudaStream_t sm = static_cast<cudaStream_t>(main);
  const size_t xb = (size_t)cfg->T * cfg->H * 2, lb = (size_t)cfg->T * cfg->E * 4;
  void* xd = at<void>(ws, L.x_stage);
  float* ld = at<float>(ws, L.logits_stage);
  void* od = at<void>(ws, L.out_stage);
  cudaError_t e = cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, sm);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ld, logits_host, lb, cudaMemcpyHostToDevice, sm);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st = moe_layer_forward(h, cfg, w, xd, nullptr, ld, od, ws, ws_bytes, main, side);
  if (st != MOE_OK) return st;
  e = cudaMemcpyAsync(out_host, od, xb, cudaMemcpyDeviceToHost, sm);
  if (e == cudaSuccess) e = cudaStreamSynchronize(sm);
  return cuda_status(e);
}

MOE_API moe_status_t moe_get_device_status(moe_handle_t h, int* code, moe_stream_t stream) {
  if (!code) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->status, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  if (v == 0) return MOE_OK;
  return (v >= MOE_DEV_BAD_EXPERT_ID) ? MOE_ERR_INVALID_ARG : MOE_ERR_DEVICE_TIMEOUT;
}

MOE_API moe_status_t moe_read_stage_times(moe_handle_t h, float* ms, int* n_calls) {
  if (!h || !ms || !n_calls) return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  for (int i = 0; i < MOE_NUM_STAGES; ++i) ms[i] = -1.0f;
  const int n = h->t_calls < kTimingRing ? h->t_calls : kTimingRing;
  *n_calls = n;
  if (n == 0 || !h->tev) return MOE_OK;
  double sum[MOE_NUM_STAGES] = {};
  int nsh = 0;
  for (int c = 0; c < n; ++c) {
    const int slot = (h->t_calls - n + c) % kTimingRing;
    cudaEvent_t* ev = h->tev + slot * kEventsPerCall;
    if (cudaEventSynchronize(ev[5]) != cudaSuccess) return MOE_ERR_CUDA;
    static const int pairs[5][2] = {{0, 1}, {1, 2}, {2, 3}, {3, 4}, {4, 5}};
    for (int sidx = 0; sidx < 5; ++sidx) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ev[pairs[sidx][0]], ev[pairs[sidx][1]]) != cudaSuccess)
        return MOE_ERR_CUDA;
      sum[sidx] += t;
    }
    float tot = 0.f;
    if (cudaEventElapsedTime(&tot, ev[0], ev[5]) != cudaSuccess) return MOE_ERR_CUDA;
    sum[MOE_STAGE_TOTAL] += tot;
    if (h->t_shared[slot]) {
      float t = 0.f;
      if (cudaEventSynchronize(ev[7]) != cudaSuccess ||
          cudaEventElapsedTime(&t, ev[6], ev[7]) != cudaSuccess)
        return MOE_ERR_CUDA;
      sum[MOE_STAGE_SHARED] += t;
      ++nsh;
    }
  }
  for (int i = 0; i < MOE_NUM_STAGES; ++i) {
    if (i == MOE_STAGE_SHARED) ms[i] = nsh ? (float)(sum[i] / nsh) : -1.0f;
    else ms[i] = (float)(sum[i] / n);
  }
  h->t_calls = 0;
  return MOE_OK;
}

MOE_API moe_status_t moe_selftest_wait_timeout(moe_handle_t h, moe_stream_t stream) {
  moe_status_t st = check_handle(h);
  if (st != MOE_OK) return st;
  return cuda_status(launch_selftest_wait(h->status, h->wait_limit_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
