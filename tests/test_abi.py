"""The C-ABI library loads and exports every entry point include/moe.h declares,
and its host-side argument checks answer without a GPU (no compute calls)."""
import ctypes

import pytest

import routed_expert_ffn_04_gb300 as moe


@pytest.fixture(scope="module")
def lib():
    return moe.load(build_if_missing=True)


def test_exports_every_declared_symbol(lib):
    names = moe.exported_names()
    assert len(names) >= 15
    for n in ["moe_route", "moe_permute", "moe_grouped_swiglu_gemm", "moe_combine", "moe_layer_forward"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert moe.status_string(moe.MOE_OK) == "ok"
    assert "workspace" in moe.status_string(moe.MOE_ERR_WORKSPACE)


def _cfg(**kw):
    d = dict(T=64, H=4096, E=192, K=8, I=1536, I_shared=1536, scaling=2.826)
    d.update(kw)
    return moe.make_config(**d)


def test_workspace_size_covers_the_buffers(lib):
    n = moe.workspace_size(_cfg())
    T, H, K, I = 64, 4096, 8, 1536
    TK = T * K
    assert n >= TK * H * 2 + TK * I * 2 + TK * H * 4 + T * H * 4
    assert moe.workspace_size(_cfg(T=128)) > n
    assert moe.grouped_gemm_workspace_size(512, 4096, 1536) >= 512 * 1536 * 2
    # MXFP8: h codes, plus scale atoms of h and of a with one 128-row block of slack per group.
    mx1 = moe.grouped_gemm_workspace_size(512, 4096, 1536, moe.MOE_MXFP8_E4M3)
    assert mx1 >= 512 * 1536 + (512 // 128 + 1) * (1536 + 4096) // 32 * 128
    mx8 = moe.grouped_gemm_workspace_size(512, 4096, 1536, moe.MOE_MXFP8_E4M3, num_groups=8)
    assert mx8 - mx1 >= 7 * (1536 + 4096) // 32 * 128


def test_mx_config_needs_whole_scale_atoms(lib):
    n = ctypes.c_size_t(0)
    for bad in (dict(H=4032), dict(I=1472), dict(I_shared=64)):
        c = _cfg(dtype=moe.MOE_MXFP8_E4M3, **bad)
        assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(ctypes.byref(_cfg(dtype=moe.MOE_MXFP8_E4M3)), ctypes.byref(n)) == moe.MOE_OK


def test_w4a8_weights_need_32_byte_alignment(lib):
    P = ctypes.c_void_p
    args = lambda wg: (None, 1, 128, 256, 128, moe.MOE_MXFP4_W4A8, P(256), P(256), None, P(wg), P(512), P(512),
                       P(256), None, P(256), P(256), P(256), 1 << 30, None)
    # Packed E2M1 weights at a 16- but not 32-byte-aligned address: rejected before any launch.
    assert lib.moe_grouped_swiglu_gemm(*args(528)) == moe.MOE_ERR_INVALID_ARG
    # Aligned: passes the argument checks and stops at the null handle (also INVALID_ARG), so
    # check the workspace path instead: a too-small workspace is reported as such.
    small = list(args(512))
    small[17] = 16
    assert lib.moe_grouped_swiglu_gemm(*small) == moe.MOE_ERR_WORKSPACE


def test_pack_mx_scales_argument_checks(lib):
    P = ctypes.c_void_p
    # cols not a multiple of 128, rows not a multiple of 128 (single) or 64 (pair), misaligned pointer.
    assert lib.moe_pack_mx_scales(None, P(256), None, 128, 96, P(256), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_mx_scales(None, P(256), None, 64, 128, P(256), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_mx_scales(None, P(256), P(512), 96, 128, P(256), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_pack_mx_scales(None, P(260), None, 128, 128, P(256), None) == moe.MOE_ERR_INVALID_ARG
    # Valid sizes with a null handle: rejected as an argument, before any launch.
    assert lib.moe_pack_mx_scales(None, P(256), P(512), 64, 128, P(256), None) == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(K=0), dict(K=9, E=8), dict(E=2048, K=8), dict(H=100), dict(I=96),
                                 dict(I_shared=32), dict(K=33, E=64), dict(T=-1), dict(T=1 << 28)])
def test_bad_configs_rejected_before_any_launch(lib, bad):
    n = ctypes.c_size_t(0)
    rc = lib.moe_workspace_size(ctypes.byref(_cfg(**bad)), ctypes.byref(n))
    assert rc == moe.MOE_ERR_INVALID_ARG


def test_null_handle_and_pointers_rejected(lib):
    cfg = _cfg()
    P = ctypes.c_void_p
    # Null handle with valid-looking pointers: rejected without touching CUDA.
    rc = lib.moe_route(None, ctypes.byref(cfg), P(4096), P(4096), P(4096), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # Misaligned pointer.
    rc = lib.moe_route(None, ctypes.byref(cfg), P(4100), P(4096), P(4096), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # Null logits.
    rc = lib.moe_route(None, ctypes.byref(cfg), None, P(4096), P(4096), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    rc = lib.moe_combine(None, ctypes.byref(cfg), None, P(16), P(16), None, P(16), None)
    assert rc == moe.MOE_ERR_INVALID_ARG


def test_small_workspace_rejected(lib):
    cfg = _cfg()
    w = moe.Weights()
    for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        setattr(w, k, 1 << 20)
    need = moe.workspace_size(cfg)
    P = ctypes.c_void_p
    rc = lib.moe_layer_forward(None, ctypes.byref(cfg), ctypes.byref(w), P(1 << 20), None, P(1 << 20), P(1 << 20),
                               P(1 << 20), need - 256, None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    # Pre-quantised activations (x_scale_or_null) only exist in the MX modes.
    rc = lib.moe_layer_forward(None, ctypes.byref(cfg), ctypes.byref(w), P(1 << 20), P(1 << 20), P(1 << 20),
                               P(1 << 20), P(1 << 20), need, None, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    rc = lib.moe_grouped_swiglu_gemm(None, 4, 100, 256, 128, 0, P(256), None, P(256), P(256), P(256), P(256),
                                     None, None, None, P(256), P(256), 10, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    rc = lib.moe_grouped_swiglu_gemm(None, 0, 100, 256, 128, 0, P(256), None, P(256), P(256), P(256), P(256),
                                     None, None, None, P(256), P(256), 1 << 30, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # offsets == NULL is only valid for a single group.
    rc = lib.moe_grouped_swiglu_gemm(None, 2, 100, 256, 128, 0, P(256), None, None, P(256), P(256), P(256),
                                     None, None, None, P(256), P(256), 1 << 30, None)
    assert rc == moe.MOE_ERR_INVALID_ARG


def test_tile_mxfp4_argument_checks(lib):
    P = ctypes.c_void_p
    # rows % 128, cols % 128 and distinct buffers are checked before the handle.
    assert lib.moe_tile_mxfp4_weights(None, P(256), None, 64, 256, P(4096), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_tile_mxfp4_weights(None, P(256), None, 128, 192, P(4096), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_tile_mxfp4_weights(None, P(256), None, 128, 256, P(256), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_tile_mxfp4_weights(None, P(256), P(512), 128, 256, P(512), None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_tile_mxfp4_weights(None, P(256), P(512), 128, 256, P(4096), None) == moe.MOE_ERR_INVALID_ARG


def test_option_validation(lib):
    assert lib.moe_set_option(None, 0, 1) == moe.MOE_ERR_INVALID_ARG
