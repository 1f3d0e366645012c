"""Python binding of the GB300 MoE FFN layer library (libmoe_gb300.so).

Argument marshalling only: every step runs in the CUDA kernels behind the C
ABI of include/moe.h. PyTorch provides device memory and streams. The binding
refuses to run when the compiled library is missing; there is no CPU path.

Names follow the C ABI: route, permute, grouped_swiglu_gemm, combine,
quantize_mxfp8, quantize_mxfp4, pack_mx_scales, layer_forward, layer_forward_host.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import _build

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE_TIMEOUT = range(6)
MOE_BF16, MOE_MXFP8_E4M3, MOE_MXFP4_W4A8 = 0, 1, 2
DTYPES = {"bf16": MOE_BF16, "mxfp8": MOE_MXFP8_E4M3, "mxfp4": MOE_MXFP4_W4A8}
(MOE_OPT_GEMM_MODE, MOE_OPT_STAGE_TIMING, MOE_OPT_WAIT_LIMIT_US, MOE_OPT_SHARED_FOLD, MOE_OPT_SHARED_SMS,
 MOE_OPT_GATHER_A, MOE_OPT_MX_TILE) = 0, 1, 2, 3, 4, 5, 6
STAGES = ["route", "permute", "gemm_gate_up", "gemm_down", "combine", "shared", "total"]
DEV_TIMEOUT_SELFTEST = 4

_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int), ("K", ctypes.c_int),
                ("I", ctypes.c_int), ("I_shared", ctypes.c_int), ("scaling", ctypes.c_float),
                ("route_norm", ctypes.c_int), ("dtype", ctypes.c_int)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
                 "ws_gate", "ws_up", "ws_down", "ss_gate", "ss_up", "ss_down")]


def exported_names() -> list[str]:
    """Entry points declared in include/moe.h (MOE_API functions)."""
    text = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)


def load(build_if_missing: bool = False):
    """Load the compiled library; raise if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        if build_if_missing:
            _build.build()
        else:
            raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    PS = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "moe_create": [I, ctypes.POINTER(P)],
        "moe_destroy": [P],
        "moe_set_option": [P, I, I],
        "moe_workspace_size": [P, PS],
        "moe_route": [P, P, P, P, P, P],
        "moe_permute_workspace_size": [P, PS],
        "moe_permute": [P, P, P, P, P, P, P, P, P, P, P, P, S, P],
        "moe_grouped_gemm_workspace_size": [I, I, I, I, I, PS],
        "moe_grouped_swiglu_gemm": [P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, S, P],
        "moe_combine": [P, P, P, P, P, P, P, P],
        "moe_quantize_mxfp8": [P, P, ctypes.c_int64, I, P, P, P],
        "moe_quantize_mxfp4": [P, P, ctypes.c_int64, I, P, P, P],
        "moe_tile_mxfp4_weights": [P, P, P, ctypes.c_int64, I, P, P],
        "moe_pack_mx_scales": [P, P, P, ctypes.c_int64, I, P, P],
        "moe_layer_forward": [P, P, P, P, P, P, P, P, S, P, P],
        "moe_layer_forward_host": [P, P, P, P, P, P, P, S, P, P],
        "moe_get_device_status": [P, ctypes.POINTER(I), P],
        "moe_read_stage_times": [P, ctypes.POINTER(F), ctypes.POINTER(I)],
        "moe_selftest_wait_timeout": [P, P],
        "moe_permute_static_scratch": [P, P, P, P, P, P, P, P, P, P, P, P],
        "moe_gate_route": [P, P, P, P, P, P, P, P],
        "moe_layer_forward_gated": [P, P, P, P, P, P, P, S, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.moe_status_string.argtypes = [I]
    lib.moe_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(s: int) -> str:
    return load().moe_status_string(int(s)).decode()


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoEError(rc, what)


def _p(t):
    """Device/host pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(s):
    if s is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(s.cuda_stream)


def make_config(T, H, E, K, I, I_shared, scaling, route_norm=True, dtype=MOE_BF16) -> Config:
    return Config(int(T), int(H), int(E), int(K), int(I), int(I_shared), float(scaling), int(bool(route_norm)), int(dtype))


def workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def permute_workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_permute_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_permute_workspace_size")
    return n.value


def grouped_gemm_workspace_size(rows: int, H: int, I: int, dtype: int = MOE_BF16, num_groups: int = 1) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_grouped_gemm_workspace_size(int(rows), int(num_groups), int(H), int(I), int(dtype),
                                                  ctypes.byref(n)), "moe_grouped_gemm_workspace_size")
    return n.value


class Handle:
    """Owns a moe_handle_t (device, SM count, status word, events)."""

    def __init__(self, device: int | None = None):
        lib = load()
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        h = ctypes.c_void_p()
        _check(lib.moe_create(self.device, ctypes.byref(h)), "moe_create")
        self._h = h

    @property
    def ptr(self):
        return self._h

    def close(self):
        if self._h:
            load().moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, opt: int, value: int):
        _check(load().moe_set_option(self._h, int(opt), int(value)), "moe_set_option")

    def device_status(self, stream=None) -> int:
        code = ctypes.c_int(0)
        rc = load().moe_get_device_status(self._h, ctypes.byref(code), _stream(stream))
        if rc not in (MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_INVALID_ARG):
            _check(rc, "moe_get_device_status")
        return code.value

    def stage_times(self) -> tuple[dict, int]:
        ms = (ctypes.c_float * 7)()
        n = ctypes.c_int(0)
        _check(load().moe_read_stage_times(self._h, ms, ctypes.byref(n)), "moe_read_stage_times")
        return {k: ms[i] for i, k in enumerate(STAGES)}, n.value

    def selftest_wait_timeout(self, stream=None):
        _check(load().moe_selftest_wait_timeout(self._h, _stream(stream)), "moe_selftest_wait_timeout")


def route(h: Handle, cfg: Config, logits, topk_idx, topk_w, stream=None):
    _check(load().moe_route(h.ptr, ctypes.byref(cfg), _p(logits), _p(topk_idx), _p(topk_w), _stream(stream)), "moe_route")


def permute(h: Handle, cfg: Config, x, topk_idx, counts, offsets, perm_src, flat_to_perm, x_perm, ws,
            x_scale=None, x_perm_scale=None, stream=None):
    _check(load().moe_permute(h.ptr, ctypes.byref(cfg), _p(x), _p(x_scale), _p(topk_idx), _p(counts), _p(offsets),
                              _p(perm_src), _p(flat_to_perm), _p(x_perm), _p(x_perm_scale), _p(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_permute")


def permute_static_scratch(h: Handle, cfg: Config, x, topk_idx, counts, offsets, perm_src, flat_to_perm, x_perm,
                           x_scale=None, x_perm_scale=None, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate: the
    histogram lives in a fixed 1 MiB array inside the library (see moe.h)."""
    _check(load().moe_permute_static_scratch(h.ptr, ctypes.byref(cfg), _p(x), _p(x_scale), _p(topk_idx), _p(counts),
                                             _p(offsets), _p(perm_src), _p(flat_to_perm), _p(x_perm),
                                             _p(x_perm_scale), _stream(stream)), "moe_permute_static_scratch")


def grouped_swiglu_gemm(h: Handle, a, offsets, w_gate, w_up, w_down, y, ws, *, num_groups: int, H: int, I: int,
                        dtype: int = MOE_BF16, a_scale=None, s_gate=None, s_up=None, s_down=None, stream=None):
    rows = a.shape[0]
    _check(load().moe_grouped_swiglu_gemm(h.ptr, int(num_groups), int(rows), int(H), int(I), int(dtype), _p(a),
                                          _p(a_scale), _p(offsets), _p(w_gate), _p(w_up), _p(w_down), _p(s_gate),
                                          _p(s_up), _p(s_down), _p(y), _p(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)), "moe_grouped_swiglu_gemm")


def combine(h: Handle, cfg: Config, y_perm, topk_w, flat_to_perm, shared_out, out, stream=None):
    _check(load().moe_combine(h.ptr, ctypes.byref(cfg), _p(y_perm), _p(topk_w), _p(flat_to_perm), _p(shared_out),
                              _p(out), _stream(stream)), "moe_combine")


def quantize_mxfp8(h: Handle, x, q, scale, stream=None):
    rows = x.numel() // x.shape[-1]
    _check(load().moe_quantize_mxfp8(h.ptr, _p(x), int(rows), int(x.shape[-1]), _p(q), _p(scale), _stream(stream)),
           "moe_quantize_mxfp8")


def quantize_mx(h: Handle, t, stream=None):
    """MXFP8 codes (uint8, same shape) and E8M0 scales (uint8, last dim / 32) of a bf16 tensor."""
    q = torch.empty(t.shape, dtype=torch.uint8, device=t.device)
    sc = torch.empty(t.shape[:-1] + (t.shape[-1] // 32,), dtype=torch.uint8, device=t.device)
    quantize_mxfp8(h, t, q, sc, stream=stream)
    return q, sc


def quantize_mxfp4(h: Handle, x, q, scale, stream=None):
    rows = x.numel() // x.shape[-1]
    _check(load().moe_quantize_mxfp4(h.ptr, _p(x), int(rows), int(x.shape[-1]), _p(q), _p(scale), _stream(stream)),
           "moe_quantize_mxfp4")


def quantize_mx4(h: Handle, t, stream=None):
    """MXFP4 packed E2M1 codes (uint8, last dim / 2) and E8M0 scales (uint8, last dim / 32) of a bf16 tensor."""
    q = torch.empty(t.shape[:-1] + (t.shape[-1] // 2,), dtype=torch.uint8, device=t.device)
    sc = torch.empty(t.shape[:-1] + (t.shape[-1] // 32,), dtype=torch.uint8, device=t.device)
    quantize_mxfp4(h, t, q, sc, stream=stream)
    return q, sc


def quantize_weights_mx(h: Handle, w: dict, stream=None, w4: bool = False) -> dict:
    """MX form of a bf16 weight dict: w_* -> E4M3 codes (w4: routed w_* -> packed
    E2M1 codes, the W4A8 recipe; the shared ws_* stay E4M3), s_* / ss_* ->
    row-major scales."""
    out = {}
    for k, v in w.items():
        q, sc = (quantize_mx4 if (w4 and k.startswith("w_")) else quantize_mx)(h, v, stream=stream)
        out[k] = q
        out[("ss_" + k[3:]) if k.startswith("ws_") else ("s_" + k[2:])] = sc
    return out


def pack_mx_scales(h: Handle, scale0, scale1=None, stream=None):
    """Scale atoms (moe_pack_mx_scales) of row-major E8M0 scales [..., cols/32]:
    of scale0 alone, or of the gate (scale0) / up (scale1) pair."""
    rows = scale0.numel() // scale0.shape[-1]
    cols = scale0.shape[-1] * 32
    out = torch.empty(scale0.numel() * (2 if scale1 is not None else 1), dtype=torch.uint8, device=scale0.device)
    _check(load().moe_pack_mx_scales(h.ptr, _p(scale0), _p(scale1), int(rows), int(cols), _p(out), _stream(stream)),
           "moe_pack_mx_scales")
    return out


def tile_mxfp4(h: Handle, q0, q1=None, stream=None):
    """Tile order (moe_tile_mxfp4_weights) of packed E2M1 codes [..., rows, cols/2]:
    of q0 alone (same shape), or of the gate (q0) / up (q1) pair (twice the
    rows)."""
    rows = q0.numel() // q0.shape[-1]
    shape = q0.shape if q1 is None else q0.shape[:-2] + (2 * q0.shape[-2], q0.shape[-1])
    out = torch.empty(shape, dtype=torch.uint8, device=q0.device)
    _check(load().moe_tile_mxfp4_weights(h.ptr, _p(q0), _p(q1), int(rows), int(q0.shape[-1] * 2), _p(out),
                                         _stream(stream)), "moe_tile_mxfp4_weights")
    return out


def pack_weights_mx(h: Handle, mx: dict, stream=None) -> dict:
    """Codes + row-major scales (quantize_weights_mx) -> the weight form the
    MX layer takes: s_gate / ss_gate = gate+up atoms, s_down / ss_down =
    down atoms, s_up / ss_up dropped; packed E2M1 routed codes (W4A8) in tile
    order: w_gate = the gate/up pair, w_up dropped, w_down alone."""
    out = {k: v for k, v in mx.items() if not k.startswith("s")}
    wg, sg = mx.get("w_gate"), mx.get("s_gate")
    if wg is not None and sg is not None and wg.shape[-1] * 2 == sg.shape[-1] * 32:  # packed E2M1
        out["w_gate"] = tile_mxfp4(h, wg, mx["w_up"], stream=stream)
        out["w_up"] = None
        out["w_down"] = tile_mxfp4(h, mx["w_down"], stream=stream)
    for p in ("s_", "ss_"):
        if mx.get(p + "gate") is None:
            continue
        out[p + "gate"] = pack_mx_scales(h, mx[p + "gate"], mx[p + "up"], stream=stream)
        out[p + "down"] = pack_mx_scales(h, mx[p + "down"], stream=stream)
    return out


def gate_route(h: Handle, cfg: Config, x, w_router, topk_idx, topk_w, logits_out=None, stream=None):
    """Gating projection + routing (fused in one kernel when E <= 256)."""
    _check(load().moe_gate_route(h.ptr, ctypes.byref(cfg), _p(x), _p(w_router), _p(logits_out), _p(topk_idx),
                                 _p(topk_w), _stream(stream)), "moe_gate_route")


def layer_forward_gated(h: Handle, cfg: Config, weights: Weights, w_router, x, out, ws, main=None, side=None):
    side_p = ctypes.c_void_p(side.cuda_stream) if side is not None else None
    _check(load().moe_layer_forward_gated(h.ptr, ctypes.byref(cfg), ctypes.byref(weights), _p(w_router), _p(x),
                                          _p(out), _p(ws), ws.numel() * ws.element_size(), _stream(main), side_p),
           "moe_layer_forward_gated")


def make_weights(w: dict) -> Weights:
    ws = Weights()
    for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down", "s_gate", "s_up", "s_down",
              "ss_gate", "ss_up", "ss_down"):
        t = w.get(k)
        setattr(ws, k, t.data_ptr() if t is not None else None)
    return ws


def layer_forward(h: Handle, cfg: Config, weights: Weights, x, logits, out, ws, main=None, side=None,
                  x_scale=None):
    """x_scale: E8M0 scales [T, H/32] when x already holds MXFP8 E4M3 codes (MX configs only)."""
    side_p = ctypes.c_void_p(side.cuda_stream) if side is not None else None
    _check(load().moe_layer_forward(h.ptr, ctypes.byref(cfg), ctypes.byref(weights), _p(x), _p(x_scale), _p(logits),
                                    _p(out), _p(ws), ws.numel() * ws.element_size(), _stream(main), side_p),
           "moe_layer_forward")


def layer_forward_host(h: Handle, cfg: Config, weights: Weights, x_host, logits_host, out_host, ws, main=None,
                       side=None):
    side_p = ctypes.c_void_p(side.cuda_stream) if side is not None else None
    _check(load().moe_layer_forward_host(h.ptr, ctypes.byref(cfg), ctypes.byref(weights), _p(x_host),
                                         _p(logits_host), _p(out_host), _p(ws), ws.numel() * ws.element_size(),
                                         _stream(main), side_p), "moe_layer_forward_host")


class MoELayer:
    """Convenience owner of a handle, workspace and side stream for one shape."""

    def __init__(self, shape, weights: dict, device=None, side_stream=True):
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.shape = shape
        self.cfg = make_config(shape.T, shape.H, shape.E, shape.K, shape.I, shape.I_shared, shape.scaling,
                               shape.route_norm, DTYPES[shape.dtype])
        self.handle = Handle(self.device.index)
        self.ws = torch.empty(workspace_size(self.cfg), dtype=torch.uint8, device=self.device)
        if shape.dtype in ("mxfp8", "mxfp4"):
            if weights["w_gate"].dtype != torch.uint8:
                weights = quantize_weights_mx(self.handle, weights, w4=shape.dtype == "mxfp4")
            if weights.get("s_up") is not None:  # row-major scales -> scale atoms
                weights = pack_weights_mx(self.handle, weights)
            torch.cuda.synchronize(self.device)
        self.weights_t = weights
        self.weights = make_weights(weights)
        self.side = torch.cuda.Stream(device=self.device) if side_stream else None

    def __call__(self, x, logits, out=None, main=None, x_scale=None):
        """x: [T, H] bf16, or (MX layers, with x_scale) MXFP8 E4M3 codes with their E8M0 scales."""
        if out is None:
            out = torch.empty((self.shape.T, self.shape.H), dtype=torch.bfloat16, device=self.device)
        layer_forward(self.handle, self.cfg, self.weights, x, logits, out, self.ws, main=main, side=self.side,
                      x_scale=x_scale)
        return out
