"""GPU parity of the CTA-pair grouped GEMM (MOE_OPT_GEMM_MODE = 3: weight rows
as the M = 256 rows of one MMA over two SMs, tokens as N) against the
oracle's per-row SwiGLU MLP: ragged group sizes (empty groups, single rows,
every N from 32 to the tile width, token chunks split across the two CTAs),
output features that end within a pair tile, and a Hy3-shaped expert.

The waits of these launches are limited to half a second, so that a
synchronisation fault shows up as a recorded timeout rather than a long
stall. Tolerance as for the other GEMM tests: y (fp32) within max-abs 2e-2
and relative L2 1e-2 of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 2e-2, 1e-2
PAIR = 3


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    h = moe.Handle(0)
    h.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 500000)
    yield h
    h.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 2000000)
    h.set_option(moe.MOE_OPT_GEMM_MODE, 0)


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
    status = handle.device_status()
    assert status == 0, f"device status {status}"
    return y.cpu().numpy()


def _check(y, ref, what):
    err = np.abs(y - ref)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(y)), what
    assert err.max() <= MAX_ABS and rel <= REL_L2, f"{what}: max {err.max():.3e} rel {rel:.3e}"


def test_one_small_group(handle):
    # The smallest case first: one group, one 256-row weight tile, N = 32.
    H, I, rows = 128, 256, 20
    a = torch.randn(rows, H, generator=torch.Generator().manual_seed(11)).to(torch.bfloat16)
    wg, wu, wd = _weights(1, H, I, 12)
    y = _run(handle, a, [0, rows], wg, wu, wd, H, I, PAIR, 1)
    _check(y, oracle.swiglu_mlp(a, wg[0], wu[0], wd[0]), "one small group")


@pytest.mark.parametrize("H,I,sizes", [
    (256, 256, [16, 0, 3, 1]),
    (256, 192, [40, 64, 65, 96, 97, 128, 129]),       # every N step; I ends with the even CTA's half
    (320, 320, [0, 1, 37, 130, 300, 0]),              # H and I end inside a pair tile
    (512, 384, [129, 127, 64, 33, 32, 31, 257, 511]),  # token chunks of 256, partial and full
])
def test_pair_gemm_matches_oracle(handle, H, I, sizes):
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    a = torch.randn(rows, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    wg, wu, wd = _weights(G, H, I, 2)
    y = _run(handle, a, offsets.tolist(), wg, wu, wd, H, I, PAIR, G)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        if r1 == r0:
            continue
        ref = oracle.swiglu_mlp(a[r0:r1], wg[g], wu[g], wd[g])
        _check(y[r0:r1], ref, f"group {g} ({r1 - r0} rows)")


def test_rows_outside_groups_untouched(handle):
    H, I = 128, 128
    offsets = [0, 50, 120]
    a = torch.randn(200, H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    wg, wu, wd = _weights(2, H, I, 6)
    y = _run(handle, a, offsets, wg, wu, wd, H, I, PAIR, 2)
    assert np.all(np.isnan(y[120:]))
    assert np.all(np.isfinite(y[:120]))


def test_pair_matches_single_sm_tiling(handle):
    # The same products in another tiling: within fp32 summation-order error.
    H, I = 512, 512
    sizes = [300, 5, 700, 0, 129]
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    a = torch.randn(int(offsets[-1]), H, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    wg, wu, wd = _weights(G, H, I, 10)
    y3 = _run(handle, a, offsets.tolist(), wg, wu, wd, H, I, PAIR, G)
    y2 = _run(handle, a, offsets.tolist(), wg, wu, wd, H, I, 2, G)
    scale = np.abs(y2).max()
    assert np.abs(y3 - y2).max() <= 2 ** -6 * scale


def test_hy3_expert_shape_one_group_many_rows(handle):
    # One Hy3-shaped expert (H=4096, I=1536) on 300 rows: token chunks of 256
    # (N = 256, then 64 for the last 44 rows).
    H, I, rows = 4096, 1536, 300
    a = torch.randn(rows, H, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    wg, wu, wd = _weights(1, H, I, 8)
    sel = np.array([0, 1, 63, 64, 127, 128, 191, 192, 255, 256, 271, 272, 299])
    ref = oracle.swiglu_mlp(a[sel], wg[0], wu[0], wd[0])
    y = _run(handle, a, [0, rows], wg, wu, wd, H, I, PAIR, 1)
    _check(y[sel], ref, "hy3 expert, pair tiling")
