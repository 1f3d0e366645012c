"""moe_permute_static_scratch: the permutation for callers that cannot call
cudaMalloc and have no workspace to give (for example a plugin inside an
engine that owns all device memory, or code that must not allocate after it
has started). Its histogram lives in a fixed array inside the library.

The GPU test calls it through the C ABI on a sequence of shapes, each twice in
a row, and checks every result against moe_permute with a caller workspace.
Up to 262144 (token, slot) pairs the permutation keeps its counters in
shared memory (one block, or a cluster of eight); above that the three-kernel
path keeps its per-warp histogram in the fixed array. The sequence covers
both, and the later large shapes (another E, another number of warps) find
the earlier ones' entries still in the array. It also covers MXFP8 and W4A8
configs, whose rows are 1-byte E4M3 codes with their E8M0 scales. The
permutation is integer work, so the bar is bit-exact, as for moe_permute
itself. This file is collected last so that a
run stopping at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import routed_expert_ffn_04_gb300 as moe
import synth

# (shape, dtype name). T*K above 262144 takes the three-kernel path, the one
# that uses the fixed array.
CASES = [
    (synth.WORKLOADS["decode"].with_(H=512, I=256, I_shared=256), "bf16"),                 # 512 pairs
    (synth.MoEShape("big_e64", T=40000, H=64, E=64, K=8, I=64, I_shared=0), "bf16"),        # 320000 pairs
    (synth.MoEShape("big_e200", T=70001, H=64, E=200, K=4, I=64, I_shared=0), "bf16"),      # 280004 pairs
    (synth.WORKLOADS["skewed"].with_(H=256, I=128, I_shared=128), "bf16"),                 # 32768 pairs, E=256
    (synth.MoEShape("mx8_big", T=33000, H=128, E=64, K=8, I=128, I_shared=0), "mxfp8"),     # 264000 pairs
    (synth.MoEShape("w4a8_big", T=90000, H=384, E=37, K=3, I=128, I_shared=0), "mxfp4"),    # 270000 pairs, H % 512 != 0
    (synth.MoEShape("mx8", T=2049, H=512, E=192, K=8, I=128, I_shared=128), "mxfp8"),      # 16392 pairs
    (synth.MoEShape("w4a8_small", T=333, H=384, E=37, K=5, I=128, I_shared=0), "mxfp4"),   # 1665 pairs
]


def _buffers(shape, mx):
    TK = max(shape.T * shape.K, 1)
    dev = "cuda"
    b = dict(counts=torch.empty(shape.E, dtype=torch.int32, device=dev),
             offsets=torch.empty(shape.E + 1, dtype=torch.int32, device=dev),
             perm_src=torch.empty(TK, dtype=torch.int32, device=dev),
             f2p=torch.empty(TK, dtype=torch.int32, device=dev))
    if mx:
        b["x_perm"] = torch.empty((TK, shape.H), dtype=torch.uint8, device=dev)
        b["x_perm_scale"] = torch.empty((TK, shape.H // 32), dtype=torch.uint8, device=dev)
    else:
        b["x_perm"] = torch.empty((TK, shape.H), dtype=torch.bfloat16, device=dev)
        b["x_perm_scale"] = None
    # Garbage in the outputs: every entry must be written by the call.
    for v in b.values():
        if v is not None:
            v.view(torch.uint8).fill_(0xA5)
    return b


def _bits(t):
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


@pytest.mark.gpu
def test_static_scratch_permute_matches_workspace_permute_twice():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    handle = moe.Handle(0)
    for n, (shape, dt) in enumerate(CASES):
        mx = dt != "bf16"
        cfg = moe.make_config(shape.T, shape.H, shape.E, shape.K, shape.I, shape.I_shared, shape.scaling,
                              dtype=moe.DTYPES[dt])
        x, logits = synth.make_activations(shape, device="cuda", seed=20 + n)
        x_scale = None
        if mx:
            x, x_scale = moe.quantize_mx(handle, x)
        idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
        w = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
        moe.route(handle, cfg, logits, idx, w)
        ref = _buffers(shape, mx)
        ws = torch.empty(moe.permute_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        moe.permute(handle, cfg, x, idx, ref["counts"], ref["offsets"], ref["perm_src"], ref["f2p"], ref["x_perm"],
                    ws, x_scale=x_scale, x_perm_scale=ref["x_perm_scale"])
        for rep in range(2):
            got = _buffers(shape, mx)
            moe.permute_static_scratch(handle, cfg, x, idx, got["counts"], got["offsets"], got["perm_src"],
                                       got["f2p"], got["x_perm"], x_scale=x_scale,
                                       x_perm_scale=got["x_perm_scale"])
            torch.cuda.synchronize()
            assert handle.device_status() == 0, (shape.name, rep)
            for k in ("counts", "offsets", "perm_src", "f2p", "x_perm", "x_perm_scale"):
                if ref[k] is None:
                    continue
                assert torch.equal(_bits(got[k]), _bits(ref[k])), (shape.name, dt, rep, k)
        # The workspace path itself is a valid counting sort of the ids.
        counts = torch.bincount(idx.flatten().long(), minlength=shape.E).int()
        assert torch.equal(ref["counts"], counts), shape.name
    handle.close()


def test_sizes_beyond_the_fixed_array_are_rejected():
    lib = moe.load(build_if_missing=True)
    # E * ceil(T*K/256) = 1024 * 4096 > 262144 entries: refused before any launch.
    cfg = moe.make_config(T=131072, H=64, E=1024, K=8, I=64, I_shared=0, scaling=1.0)
    P = ctypes.c_void_p
    rc = lib.moe_permute_static_scratch(None, ctypes.byref(cfg), P(256), None, P(256), P(256), P(256), P(256),
                                        P(256), P(256), None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    assert np.int64(1024) * 4096 > 262144


@pytest.mark.parametrize("dtype", [moe.MOE_MXFP8_E4M3, moe.MOE_MXFP4_W4A8])
def test_mx_configs_take_the_same_arguments_as_moe_permute(dtype):
    lib = moe.load(build_if_missing=True)
    P = ctypes.c_void_p
    # H = 384 is allowed for MX (a multiple of 128). With every argument valid
    # but a null handle, both calls stop only at the handle check.
    cfg = moe.make_config(T=100, H=384, E=16, K=4, I=128, I_shared=0, scaling=1.0, dtype=dtype)
    rc = lib.moe_permute_static_scratch(None, ctypes.byref(cfg), P(256), P(256), P(256), P(256), P(256), P(256),
                                        P(256), P(256), P(256), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # Missing MX scale pointers are refused for W4A8 as well as MXFP8.
    rc = lib.moe_permute_static_scratch(None, ctypes.byref(cfg), P(256), None, P(256), P(256), P(256), P(256),
                                        P(256), P(256), None, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
