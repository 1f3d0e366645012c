"""GPU parity of the weights-as-M MX GEMMs (MOE_OPT_MX_TILE = 3: 256 weight rows
as two M = 128 block-scaled MMAs against up to 64 token rows of one expert as
N; GEMM-1 pairs each gate row with its up row across TMEM lane quarters, GEMM-2
stores 256 columns of y) for MXFP8 and W4A8 weights, against the oracle's MX
SwiGLU MLP ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.2):
empty groups, single rows, groups of exactly 64 and 65 rows (a second token
chunk, whose scales sit two TMEM columns into the activation atom), groups of
several 128-row atom blocks, and the decode workload's shape at every expert's
tile edges. Also against the 128-row tiling on the same operands.

Waits are limited to half a second, so a synchronisation fault shows up as a
recorded timeout. MX bars as for the other MX tests: relative L2 <= 3e-2 and
max-abs <= 2e-2 against the oracle on the same quantised operands."""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import edge_tokens

pytestmark = pytest.mark.gpu

REL_L2_MX = 3e-2
MAX_ABS_MX = 2e-2
SWAP, NARROW = 3, 1


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    h = moe.Handle(0)
    h.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 500000)
    yield h
    h.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 2000000)
    h.set_option(moe.MOE_OPT_MX_TILE, 0)


def _check(got, ref, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(got)), what
    assert rel <= REL_L2_MX and err.max() <= MAX_ABS_MX, f"{what}: rel_l2={rel:.3e} max_abs={err.max():.3e}"


def _quantised_weights(handle, wg, wu, wd, w4):
    mw = moe.quantize_weights_mx(handle, {"w_gate": wg.cuda(), "w_up": wu.cuda(), "w_down": wd.cuda()}, w4=w4)
    return moe.pack_weights_mx(handle, mw)


def _run_gemm(handle, tile, aq, as_, offsets, pw, H, I, G, dtype):
    handle.set_option(moe.MOE_OPT_MX_TILE, tile)
    rows = aq.shape[0]
    y = torch.full((rows, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.grouped_gemm_workspace_size(rows, H, I, dtype, num_groups=G), dtype=torch.uint8,
                     device="cuda")
    moe.grouped_swiglu_gemm(handle, aq, torch.from_numpy(offsets).cuda(), pw["w_gate"], pw["w_up"], pw["w_down"], y, ws,
                            num_groups=G, H=H, I=I, dtype=dtype, a_scale=as_, s_gate=pw["s_gate"],
                            s_down=pw["s_down"])
    torch.cuda.synchronize()
    status = handle.device_status()
    assert status == 0, f"device status {status}"
    return y.cpu().numpy()


def _operands(H, I, sizes, seed):
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(int(offsets[-1]), H, generator=g).to(torch.bfloat16)
    wg, wu, wd = ((torch.randn(*sh, generator=g) * 0.02).to(torch.bfloat16) for sh in ((G, I, H), (G, I, H), (G, H, I)))
    return G, offsets, a, wg, wu, wd


def _per_group(y, offsets, a, wg, wu, wd, w4):
    q = oracle.mxfp4_quantize if w4 else oracle.mx_quantize
    xq, xs = oracle.mx_quantize(a)
    for gi in range(len(offsets) - 1):
        r0, r1 = offsets[gi], offsets[gi + 1]
        if r1 == r0:
            continue
        ref = oracle.swiglu_mlp_mx(xq[r0:r1], xs[r0:r1], q(wg[gi]), q(wu[gi]), q(wd[gi]), w4=w4)
        _check(y[r0:r1], ref, f"group {gi} ({r1 - r0} rows)")
    assert np.all(np.isnan(y[offsets[-1]:]))


@pytest.mark.parametrize("w4", [False, True])
def test_one_small_group(handle, w4):
    # The smallest case first: one group, one tile per GEMM, 3 rows (one 16-row token box).
    H, I = 256, 128
    G, offsets, a, wg, wu, wd = _operands(H, I, [3], 31)
    dtype = moe.MOE_MXFP4_W4A8 if w4 else moe.MOE_MXFP8_E4M3
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    pw = _quantised_weights(handle, wg, wu, wd, w4)
    y = _run_gemm(handle, SWAP, aq, as_, offsets, pw, H, I, G, dtype)
    _per_group(y, offsets, a, wg, wu, wd, w4)


@pytest.mark.parametrize("w4", [False, True])
@pytest.mark.parametrize("H,I,sizes", [
    (256, 128, [16, 0, 3, 1, 17, 33]),            # one chunk per group, one to three token boxes
    (512, 384, [0, 1, 64, 65, 0, 2]),             # a chunk of exactly 64 rows; a second chunk of one row
    (256, 640, [127, 128, 129, 5, 300]),          # odd and even chunks over several activation atom blocks
])
def test_swap_gemm_matches_oracle(handle, w4, H, I, sizes):
    G, offsets, a, wg, wu, wd = _operands(H, I, sizes, 32)
    dtype = moe.MOE_MXFP4_W4A8 if w4 else moe.MOE_MXFP8_E4M3
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    pw = _quantised_weights(handle, wg, wu, wd, w4)
    y = _run_gemm(handle, SWAP, aq, as_, offsets, pw, H, I, G, dtype)
    _per_group(y, offsets, a, wg, wu, wd, w4)


@pytest.mark.parametrize("w4", [False, True])
def test_swap_matches_narrow_tiling(handle, w4):
    H, I = 512, 512
    G, offsets, a, wg, wu, wd = _operands(H, I, [3, 70, 0, 1, 129, 8], 33)
    dtype = moe.MOE_MXFP4_W4A8 if w4 else moe.MOE_MXFP8_E4M3
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    pw = _quantised_weights(handle, wg, wu, wd, w4)
    ys = _run_gemm(handle, SWAP, aq, as_, offsets, pw, H, I, G, dtype)
    yn = _run_gemm(handle, NARROW, aq, as_, offsets, pw, H, I, G, dtype)
    # h is re-quantised to E4M3: an fp32 summation-order difference can flip a
    # code, so compare y within a few E4M3 steps of h, not bit for bit.
    scale = np.abs(yn).max()
    assert np.abs(ys - yn).max() <= 2 ** -5 * scale


def test_gemm1_only_when_gemm2_cannot_swap(handle):
    # H % 256 != 0: GEMM-1 takes the weights-as-M tiling, GEMM-2 the 128-row
    # kernel, which reads the h scale atoms GEMM-1 wrote.
    H, I = 384, 256
    G, offsets, a, wg, wu, wd = _operands(H, I, [5, 0, 66, 2], 34)
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    pw = _quantised_weights(handle, wg, wu, wd, True)
    y = _run_gemm(handle, SWAP, aq, as_, offsets, pw, H, I, G, moe.MOE_MXFP4_W4A8)
    _per_group(y, offsets, a, wg, wu, wd, True)


def _w_oracle(w, w4):
    return {k: (oracle.mxfp4_quantize(v.cpu()) if (w4 and k.startswith("w_")) else oracle.mx_quantize(v.cpu()))
            for k, v in w.items()}


@pytest.mark.parametrize("dtype", ["mxfp8", "mxfp4"])
def test_swap_layer_ragged_shape(handle, dtype):
    shape = synth.MoEShape("mxs", T=21, H=512, E=13, K=3, I=256, I_shared=128, dtype=dtype)
    x, logits = synth.make_activations(shape, seed=8)
    w = synth.make_weights(shape, seed=8)
    layer = moe.MoELayer(shape, {k: v.cuda() for k, v in w.items()}, device=0)
    layer.handle.set_option(moe.MOE_OPT_MX_TILE, SWAP)
    out = layer(x.cuda(), logits.cuda())
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    w4 = dtype == "mxfp4"
    ref = oracle.layer_forward_mx(x, logits, _w_oracle(w, w4), K=shape.K, scaling=shape.scaling, w4=w4)
    _check(out.float().cpu().numpy(), ref, f"ragged {dtype}")


@pytest.mark.parametrize("dtype", ["mxfp8", "mxfp4"])
def test_swap_layer_decode_shape_tile_edges(handle, dtype):
    shape = synth.WORKLOADS["decode"].with_(dtype=dtype)
    x, logits = synth.make_activations(shape, device="cuda", seed=0)
    w = synth.make_weights(shape, device="cuda", seed=0)
    layer = moe.MoELayer(shape, w, device=0)
    layer.handle.set_option(moe.MOE_OPT_MX_TILE, SWAP)
    out = layer(x, logits)
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    w4 = dtype == "mxfp4"
    ridx, _ = oracle.route(logits.cpu().numpy(), shape.K, shape.scaling)
    tokens = edge_tokens(ridx, shape.E, sample=16, seed=6)
    ref = oracle.layer_forward_mx(x.cpu(), logits.cpu(), _w_oracle(w, w4), K=shape.K, scaling=shape.scaling,
                                  tokens=tokens, w4=w4)
    _check(out.float().cpu().numpy()[tokens], ref, f"decode shape {dtype}, weights as M")


def test_more_tiles_per_cta_than_the_prologue_list(handle):
    # A CTA decodes its first 64 tiles once in the prologue and searches the
    # group table for the rest. 64 groups of 320 rows (five 64-row chunks) x 32
    # weight tiles of I = 4096 give 10240 GEMM-1 tiles, about 67 per CTA on 152
    # SMs; the last groups' tiles are the ones past the list.
    H, I, G = 256, 4096, 64
    sizes = [320] * G
    G, offsets, a, wg, wu, wd = _operands(H, I, sizes, 35)
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    pw = _quantised_weights(handle, wg, wu, wd, False)
    y = _run_gemm(handle, SWAP, aq, as_, offsets, pw, H, I, G, moe.MOE_MXFP8_E4M3)
    xq, xs = oracle.mx_quantize(a)
    q = oracle.mx_quantize
    for gi in (0, G - 2, G - 1):
        r0, r1 = offsets[gi], offsets[gi + 1]
        ref = oracle.swiglu_mlp_mx(xq[r0:r1], xs[r0:r1], q(wg[gi]), q(wu[gi]), q(wd[gi]))
        _check(y[r0:r1], ref, f"group {gi}")


@pytest.mark.parametrize("G,fallback", [(512, False), (513, True)])
def test_group_table_limit(handle, G, fallback):
    # The weights-as-M kernels hold up to 512 groups in shared memory: 512 run
    # them, 513 take the 128-row kernels (E4M3 weights), same results either way.
    H, I = 256, 128
    sizes = [0] * G
    for gi, n in ((0, 3), (100, 1), (257, 70), (G - 2, 5), (G - 1, 33)):
        sizes[gi] = n
    G, offsets, a, wg, wu, wd = _operands(H, I, sizes, 36)
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    pw = _quantised_weights(handle, wg, wu, wd, False)
    y = _run_gemm(handle, SWAP, aq, as_, offsets, pw, H, I, G, moe.MOE_MXFP8_E4M3)
    _per_group(y, offsets, a, wg, wu, wd, False)
