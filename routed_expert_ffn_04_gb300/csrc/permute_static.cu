// The permutation step (counting sort + row gather) for callers that cannot
// allocate device memory and cannot hand the library a workspace, such as a
// plugin living inside an engine that owns every device allocation and
// exposes no allocator to it, or code that must not allocate once it has
// started (a fixed memory budget, no allocator calls on the hot path).
//
// It runs the same kernels as moe_permute. The only difference is where the
// per-warp histogram lives: in g_permute_scratch below, a fixed array in the
// library's own device memory, instead of a caller workspace. Every GPU that
// loads the library holds that array (1 MiB) until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Histogram scratch shared by every call on a device. Nothing in it needs to
// start at zero: each call writes every entry it later reads.
static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_STATIC_MAX_HIST_INTS];

struct ScratchAddr {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchAddr g_addr[kMaxDevices];

// Device address of g_permute_scratch on `device` (which must be current).
// In host code the array's name is only a host-side stand-in, so the address
// is looked up once per device and cached for the life of the process. The
// cache does not survive cudaDeviceReset (the array is re-created at a new
// address): a process that resets a device must not call this entry point
// on it again.
cudaError_t scratch_address(int device, void** out) {
  ScratchAddr& a = g_addr[device];
  std::call_once(a.once, [&a] { a.err = cudaGetSymbolAddress(&a.ptr, g_permute_scratch); });
  *out = a.ptr;
  return a.err;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" MOE_API moe_status_t moe_permute_static_scratch(
    moe_handle_t h, const moe_config_t* cfg, const void* x, const uint8_t* x_scale,
    const int32_t* topk_idx, int32_t* counts, int32_t* offsets, int32_t* perm_src,
    int32_t* flat_to_perm, void* x_perm, uint8_t* x_perm_scale, moe_stream_t stream) {
  size_t need = 0;
  moe_status_t st = moe_permute_workspace_size(cfg, &need);  // validates cfg
  if (st != MOE_OK) return st;
  // MXFP8 and W4A8 both move 1-byte E4M3 rows plus their E8M0 scales.
  const bool mx = moe::is_mx_dtype(cfg->dtype);
  const bool any = cfg->T > 0;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (any && (!x || !topk_idx || !perm_src || !flat_to_perm || !x_perm)) return MOE_ERR_INVALID_ARG;
  if (any && mx && (!x_scale || !x_perm_scale)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, topk_idx, counts, offsets, perm_src, flat_to_perm, x_perm};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (mx && (!aligned16(x_scale) || !aligned16(x_perm_scale))) return MOE_ERR_INVALID_ARG;
  // The histogram has E * ceil(T*K / 256) entries; the fixed array caps it.
  const long long nw = ((long long)cfg->T * cfg->K + 255) / 256;
  if ((long long)cfg->E * (nw > 0 ? nw : 1) > MOE_PERMUTE_STATIC_MAX_HIST_INTS)
    return MOE_ERR_WORKSPACE;
  if (!h) return MOE_ERR_INVALID_ARG;

  const int dev = moe::handle_device(h);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ERR_CUDA;
  if (cur != dev && cudaSetDevice(dev) != cudaSuccess) return MOE_ERR_CUDA;
  // The caller's current device is put back on every return below.
  auto done = [cur, dev](moe_status_t r) {
    if (cur != dev && cudaSetDevice(cur) != cudaSuccess && r == MOE_OK) r = MOE_ERR_CUDA;
    return r;
  };
  void* scratch = nullptr;
  if (scratch_address(dev, &scratch) != cudaSuccess || scratch == nullptr) return done(MOE_ERR_CUDA);

  int* status = moe::handle_status_word(h);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int TK = cfg->T * cfg->K;
  cudaError_t e = moe::launch_permute_index(topk_idx, TK, cfg->E, scratch, counts, offsets,
                                            nullptr, perm_src, flat_to_perm, status, s);
  if (e == cudaSuccess)
    e = moe::launch_scatter_rows(x, cfg->T, mx ? cfg->H : cfg->H * 2, flat_to_perm, cfg->K, TK,
                                 x_perm, status, s);
  if (e == cudaSuccess && mx)
    e = moe::launch_scatter_rows(x_scale, cfg->T, cfg->H / 32, flat_to_perm, cfg->K, TK,
                                 x_perm_scale, status, s);
  return done(e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA);
}
