"""GPU parity of the grouped SwiGLU GEMM (step 3) against the oracle's
per-row SwiGLU MLP, in both tilings, on ragged group sizes (empty groups,
single rows, partial tiles in every dimension) and on a dense single group.

Tolerance: y (fp32) vs the fp64 oracle within max-abs 2e-2 and relative L2
1e-2 (the intermediate h is rounded to bf16 on the GPU)."""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-2, 1e-2


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    return moe.Handle(0)


def _weights(G, H, I, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: (torch.randn(*s, generator=g) * 0.02).to(torch.bfloat16)
    return mk(G, I, H), mk(G, I, H), mk(G, H, I)


def _run(handle, a, offsets, wg, wu, wd, H, I, mode, G):
    rows = a.shape[0]
    handle.set_option(moe.MOE_OPT_GEMM_MODE, mode)
    y = torch.full((rows, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.grouped_gemm_workspace_size(rows, H, I), dtype=torch.uint8, device="cuda")
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int32, device="cuda")
    moe.grouped_swiglu_gemm(handle, a.cuda(), off, wg.cuda(), wu.cuda(), wd.cuda(), y, ws, num_groups=G, H=H, I=I)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    return y.cpu().numpy()


def _check(y, ref, what):
    err = np.abs(y - ref)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(y)), what
    assert err.max() <= MAX_ABS and rel <= REL_L2, f"{what}: max {err.max():.3e} rel {rel:.3e}"


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("H,I,sizes", [
    (256, 128, [16, 0, 3, 1]),
    (320, 320, [0, 1, 37, 130, 300, 0]),        # partial tiles along H, I and rows
    (512, 384, [129, 127, 64, 33, 32, 31]),
])
def test_grouped_gemm_matches_oracle(handle, mode, H, I, sizes):
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    a = torch.randn(rows, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    wg, wu, wd = _weights(G, H, I, 2)
    y = _run(handle, a, offsets.tolist(), wg, wu, wd, H, I, mode, G)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        ref = oracle.swiglu_mlp(a[r0:r1], wg[g], wu[g], wd[g])
        _check(y[r0:r1], ref, f"group {g} mode {mode}")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_dense_single_group(handle, mode):
    H, I, rows = 256, 192, 75
    a = torch.randn(rows, H, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    wg, wu, wd = _weights(1, H, I, 4)
    y = _run(handle, a, None, wg, wu, wd, H, I, mode, 1)
    _check(y, oracle.swiglu_mlp(a, wg[0], wu[0], wd[0]), f"dense mode {mode}")


def test_rows_outside_groups_untouched(handle):
    H, I = 128, 128
    sizes = [5, 7]
    offsets = [0, 5, 12]
    a = torch.randn(20, H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    wg, wu, wd = _weights(2, H, I, 6)
    y = _run(handle, a, offsets, wg, wu, wd, H, I, 0, 2)
    assert np.all(np.isnan(y[12:]))
    assert np.all(np.isfinite(y[:12]))


def test_hy3_expert_shape_one_group_many_rows(handle):
    # One Hy3-shaped expert (H=4096, I=1536) on 300 rows, both tilings.
    H, I, rows = 4096, 1536, 300
    a = torch.randn(rows, H, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    wg, wu, wd = _weights(1, H, I, 8)
    sel = np.array([0, 1, 127, 128, 255, 256, 299])
    ref = oracle.swiglu_mlp(a[sel], wg[0], wu[0], wd[0])
    for mode in (1, 2):
        y = _run(handle, a, [0, rows], wg, wu, wd, H, I, mode, 1)
        _check(y[sel], ref, f"hy3 expert mode {mode}")
