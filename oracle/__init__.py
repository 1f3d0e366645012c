"""Oracle for the sigmoid-routed top-k MoE FFN layer (TEST INFRASTRUCTURE ONLY).

A plain, slow CPU statement of the layer in double precision, written in C++
(``oracle.cpp``) and loaded here with ctypes. Only the tests, the smoke check
and the bench's CPU-baseline leg may import this package. The CUDA library
never calls it, and the two share no code.

Sources (page titles):
  [Hy3]  "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 一
         (model facts), section 8.5 (shared-expert multi-stream), section 8.2
         (MXFP8 W8A8; MXFP4 routed experts with MXFP8 activations, W4A8).
  [HyI3] "HunyuanImage-3.0 MoE 多流变体实战", 源码级实现拆解 §3 (output =
         hidden_states_mlp + combined_output).
  [OCP-MX] OCP Microscaling Formats (MX) v1.0, conversion to MX formats and
         the E4M3 / E2M1 element-format tables.

Parity is pinned for every function here by the ``-m "not gpu"`` tests
(brute force, closed forms, invariants, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``liboracle.so`` (g++ -O2 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_route.argtypes = [i, i, i, P, d, i, P, P]
            lib.oracle_gate.argtypes = [i, i, i, P, P, P]
            lib.oracle_permute.argtypes = [i, i, i, P, P, P, P, P]
            lib.oracle_swiglu_mlp.argtypes = [i, i, i, P, P, P, P, P]
            lib.oracle_layer_forward.argtypes = [i, i, i, i, i, i, d, i] + [P] * 8 + [i, P, P, P, P]
            lib.oracle_layer_forward_mx.argtypes = [i, i, i, i, i, i, i, d, i] + [P] * 14 + [i, P, P]
            lib.oracle_swiglu_mlp_mx.argtypes = [i, i, i, i] + [P] * 9
            lib.oracle_mxfp4_quantize_bf16.argtypes = [i, i, P, P, P]
            lib.oracle_mxfp4_dequantize.argtypes = [i, i, P, P, P]
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_value.restype = d
            lib.oracle_e2m1_encode.argtypes = [d]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_mx_quantize_bf16.argtypes = [i, i, P, P, P]
            lib.oracle_mx_quantize_f64.argtypes = [i, i, P, P, P]
            lib.oracle_mx_dequantize.argtypes = [i, i, P, P, P]
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = d
            lib.oracle_e4m3_encode.argtypes = [d]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_num_threads.restype = i
            lib.oracle_set_num_threads.argtypes = [i]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(a) -> np.ndarray:
    """Accept a numpy uint16 array of bf16 bit patterns, or a torch bf16 tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # local import: the oracle itself does not need torch

    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def gate(x, w_router) -> np.ndarray:
    """Router logits x w_router^T in float64 ([Hy3] section 8.5, Gating)."""
    xb, wb = _bf16_bits(x), _bf16_bits(w_router)
    T, H = xb.shape
    E = wb.shape[0]
    assert wb.shape == (E, H)
    out = np.empty((T, E), np.float64)
    _check(_load().oracle_gate(T, H, E, _ptr(xb), _ptr(wb), _ptr(out)), "gate")
    return out


def route(logits: np.ndarray, K: int, scaling: float, route_norm: bool = True):
    """Sigmoid top-k routing ([Hy3] section 一). Returns (topk_idx int32, topk_w float64)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    _check(_load().oracle_route(T, E, K, _ptr(logits), float(scaling), int(route_norm), _ptr(idx), _ptr(w)), "route")
    return idx, w


def permute(topk_idx: np.ndarray, E: int):
    """Stable expert-contiguous permutation (InitRouting, [Hy3] section 8.5).

    Returns (counts[E], offsets[E+1], perm_src[TK], flat_to_perm[TK]), all int32.
    """
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_src = np.empty(T * K, np.int32)
    flat_to_perm = np.empty(T * K, np.int32)
    _check(_load().oracle_permute(T, K, E, _ptr(topk_idx), _ptr(counts), _ptr(offsets), _ptr(perm_src), _ptr(flat_to_perm)), "permute")
    return counts, offsets, perm_src, flat_to_perm


def swiglu_mlp(x, w_gate, w_up, w_down) -> np.ndarray:
    """Dense SwiGLU MLP on bf16 rows; float64 result [R, H]."""
    x, wg, wu, wd = (_bf16_bits(a) for a in (x, w_gate, w_up, w_down))
    R, H = x.shape
    I = wg.shape[0]
    assert wg.shape == (I, H) and wu.shape == (I, H) and wd.shape == (H, I)
    y = np.empty((R, H), np.float64)
    _check(_load().oracle_swiglu_mlp(R, H, I, _ptr(x), _ptr(wg), _ptr(wu), _ptr(wd), _ptr(y)), "swiglu_mlp")
    return y


def layer_forward(x, logits, w_gate, w_up, w_down, ws_gate=None, ws_up=None, ws_down=None,
                  *, K: int, scaling: float, route_norm: bool = True, tokens=None):
    """The whole layer (float64) for `tokens` (default: all).

    Returns (out [n, H] float64, topk_idx [n, K] int32, topk_w [n, K] float64).
    """
    x = _bf16_bits(x)
    wg, wu, wd = (_bf16_bits(a) for a in (w_gate, w_up, w_down))
    logits = np.ascontiguousarray(np.asarray(logits.cpu() if hasattr(logits, "cpu") else logits), dtype=np.float32)
    T, H = x.shape
    E, I, _ = wg.shape
    if ws_gate is not None:
        sg, su, sd = (_bf16_bits(a) for a in (ws_gate, ws_up, ws_down))
        Is = sg.shape[0]
    else:
        sg = su = sd = np.zeros(1, np.uint16)
        Is = 0
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    out = np.empty((n, H), np.float64)
    idx = np.empty((n, K), np.int32)
    w = np.empty((n, K), np.float64)
    _check(_load().oracle_layer_forward(T, H, E, K, I, Is, float(scaling), int(route_norm), _ptr(x), _ptr(logits),
                                        _ptr(wg), _ptr(wu), _ptr(wd), _ptr(sg), _ptr(su), _ptr(sd),
                                        n, _ptr(tokens), _ptr(out), _ptr(idx), _ptr(w)), "layer_forward")
    return out, idx, w


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def mx_quantize(a) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8 quantisation along the last axis ([OCP-MX] conversion rule). bf16 or float64 input.

    Returns (codes uint8 [rows, cols], scales uint8 [rows, cols/32]).
    """
    lib = _load()
    if isinstance(a, np.ndarray) and a.dtype == np.float64:
        a2 = np.ascontiguousarray(a.reshape(-1, a.shape[-1]))
        fn = lib.oracle_mx_quantize_f64
    else:
        a2 = _bf16_bits(a)
        a2 = np.ascontiguousarray(a2.reshape(-1, a2.shape[-1]))
        fn = lib.oracle_mx_quantize_bf16
    rows, cols = a2.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    _check(fn(rows, cols, _ptr(a2), _ptr(q), _ptr(s)), "mx_quantize")
    lead = tuple(a.shape[:-1])
    return q.reshape(lead + (cols,)), s.reshape(lead + (cols // 32,))


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e2m1_encode(v: float) -> int:
    return int(_load().oracle_e2m1_encode(float(v)))


def mxfp4_quantize(a) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 quantisation along the last axis ([OCP-MX] rule, E2M1 elements) of a bf16 tensor.

    Returns (packed codes uint8 [..., cols/2], element 2j in the low nibble;
    scales uint8 [..., cols/32]).
    """
    a2 = _bf16_bits(a)
    a2 = np.ascontiguousarray(a2.reshape(-1, a2.shape[-1]))
    rows, cols = a2.shape
    q = np.empty((rows, cols // 2), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    _check(_load().oracle_mxfp4_quantize_bf16(rows, cols, _ptr(a2), _ptr(q), _ptr(s)), "mxfp4_quantize")
    lead = tuple(a.shape[:-1])
    return q.reshape(lead + (cols // 2,)), s.reshape(lead + (cols // 32,))


def mxfp4_dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q2 = np.ascontiguousarray(q.reshape(-1, q.shape[-1]), dtype=np.uint8)
    s2 = np.ascontiguousarray(s.reshape(-1, s.shape[-1]), dtype=np.uint8)
    rows, cols = q2.shape[0], q2.shape[1] * 2
    out = np.empty((rows, cols), np.float64)
    _check(_load().oracle_mxfp4_dequantize(rows, cols, _ptr(q2), _ptr(s2), _ptr(out)), "mxfp4_dequantize")
    return out.reshape(q.shape[:-1] + (cols,))


def mx_dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q2 = np.ascontiguousarray(q.reshape(-1, q.shape[-1]), dtype=np.uint8)
    s2 = np.ascontiguousarray(s.reshape(-1, s.shape[-1]), dtype=np.uint8)
    rows, cols = q2.shape
    out = np.empty((rows, cols), np.float64)
    _check(_load().oracle_mx_dequantize(rows, cols, _ptr(q2), _ptr(s2), _ptr(out)), "mx_dequantize")
    return out.reshape(q.shape)


def layer_forward_mx(x, logits, mx_w, *, K: int, scaling: float, route_norm: bool = True, tokens=None,
                     w4: bool = False):
    """The whole layer in MX mode (float64 out) for `tokens`.

    mx_w: dict with 'w_gate','w_up','w_down','ws_gate','ws_up','ws_down', each a
    (codes, scales) pair as returned by mx_quantize; with w4 (W4A8) the routed
    'w_*' pairs come from mxfp4_quantize instead (packed E2M1 codes).
    """
    x = _bf16_bits(x)
    logits = np.ascontiguousarray(np.asarray(logits.cpu() if hasattr(logits, "cpu") else logits), dtype=np.float32)
    T, H = x.shape
    qg, sg = mx_w["w_gate"]
    E, I = qg.shape[0], qg.shape[1]
    qs = mx_w["ws_gate"][0]
    Is = qs.shape[0]
    arrs = []
    for name in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        q, s = mx_w[name]
        arrs += [np.ascontiguousarray(q, dtype=np.uint8), np.ascontiguousarray(s, dtype=np.uint8)]
    tokens = np.arange(T, dtype=np.int32) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    out = np.empty((n, H), np.float64)
    _check(_load().oracle_layer_forward_mx(int(w4), T, H, E, K, I, Is, float(scaling), int(route_norm), _ptr(x),
                                           _ptr(logits),
                                           *[_ptr(a) for a in arrs], n, _ptr(tokens), _ptr(out)), "layer_forward_mx")
    return out


def swiglu_mlp_mx(xq: np.ndarray, xs: np.ndarray, w_gate, w_up, w_down, w4: bool = False) -> np.ndarray:
    """Dense SwiGLU MLP on MX-quantised rows with MX weights ([Hy3] section 8.2).

    xq/xs: codes [R, H] and scales [R, H/32]; w_*: (codes, scales) pairs with
    w_gate/w_up codes [I, H] and w_down codes [H, I] (w4: packed E2M1 codes
    [I, H/2] and [H, I/2] from mxfp4_quantize). Returns float64 [R, H].
    """
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=np.uint8)
    R, H = xq.shape
    I = w_gate[1].shape[0]
    arrs = []
    for q, sc in (w_gate, w_up, w_down):
        arrs += [np.ascontiguousarray(q, dtype=np.uint8), np.ascontiguousarray(sc, dtype=np.uint8)]
    y = np.empty((R, H), np.float64)
    _check(_load().oracle_swiglu_mlp_mx(int(w4), R, H, I, _ptr(xq), _ptr(xs), *[_ptr(a) for a in arrs], _ptr(y)),
           "swiglu_mlp_mx")
    return y
