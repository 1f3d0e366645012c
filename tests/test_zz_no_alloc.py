"""moe_permute_static_scratch: the permutation for callers that cannot call
cudaMalloc and have no workspace to give (for example a plugin inside an
engine that owns all device memory, or code that must not allocate after it
has started). Its histogram lives in a fixed array inside the library.

The GPU test calls it twice in a row through the C ABI and checks each result
against moe_permute with a caller workspace. The permutation is integer work,
so the bar is bit-exact, as for moe_permute itself. This file is collected
last so that a run stopping at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import routed_expert_ffn_04_gb300 as moe
import synth


def _buffers(shape):
    TK = max(shape.T * shape.K, 1)
    dev = "cuda"
    return dict(counts=torch.empty(shape.E, dtype=torch.int32, device=dev),
                offsets=torch.empty(shape.E + 1, dtype=torch.int32, device=dev),
                perm_src=torch.empty(TK, dtype=torch.int32, device=dev),
                f2p=torch.empty(TK, dtype=torch.int32, device=dev),
                x_perm=torch.empty((TK, shape.H), dtype=torch.bfloat16, device=dev))


def _cfg(shape):
    return moe.make_config(shape.T, shape.H, shape.E, shape.K, shape.I, shape.I_shared, shape.scaling)


@pytest.mark.gpu
def test_static_scratch_permute_matches_workspace_permute_twice():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    handle = moe.Handle(0)
    # Two calls in a row with different shapes: the second reuses the array
    # the first one filled.
    shapes = [synth.WORKLOADS["decode"].with_(H=512, I=256, I_shared=256),
              synth.MoEShape("ragged", T=333, H=256, E=37, K=5, I=128, I_shared=0)]
    for n, shape in enumerate(shapes):
        cfg = _cfg(shape)
        x, logits = synth.make_activations(shape, device="cuda", seed=20 + n)
        idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
        w = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
        moe.route(handle, cfg, logits, idx, w)
        ref = _buffers(shape)
        ws = torch.empty(moe.permute_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        moe.permute(handle, cfg, x, idx, ref["counts"], ref["offsets"], ref["perm_src"], ref["f2p"], ref["x_perm"], ws)
        got = _buffers(shape)
        moe.permute_static_scratch(handle, cfg, x, idx, got["counts"], got["offsets"], got["perm_src"], got["f2p"],
                                   got["x_perm"])
        torch.cuda.synchronize()
        assert handle.device_status() == 0
        for k in ("counts", "offsets", "perm_src", "f2p"):
            assert torch.equal(got[k], ref[k]), (n, k)
        assert torch.equal(got["x_perm"].view(torch.int16), ref["x_perm"].view(torch.int16)), n
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
