"""GPU parity of the W4A8 path: MXFP4 routed-expert weights (E2M1 elements,
E8M0 scale per 32 along K), MXFP8 activations and a W8A8 shared expert
("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.2), against
the oracle's W4A8 statement.

The MXFP4 quantiser is byte work and is compared bit-exactly (codes, packing
and scales). The grouped GEMM and the layer are compared with the oracle on
the same quantised operands, with the MX bars: relative L2 <= 3e-2 and
max-abs <= 2e-2 (both sides multiply the same E2M1 / E4M3 values; what
differs is fp32 accumulation and the odd E4M3 rounding flip of h).
"""
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


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    return moe.Handle(0)


def _check(got, ref, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(got)), what
    assert rel <= REL_L2_MX and err.max() <= MAX_ABS_MX, f"{what}: rel_l2={rel:.3e} max_abs={err.max():.3e}"


def test_mxfp4_quantiser_bit_exact(handle):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(193, 256, generator=g) * torch.exp(torch.randn(193, 1, generator=g) * 4)
    x[0, :32] = 0.0                                       # zero block -> scale 0, codes 0
    x[1, :32] = -0.0
    x[2, :32] = torch.tensor([0, .25, .75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4) * 2.0 ** -3  # every tie
    x[2, 5] = 6.0 * 2.0 ** -3                             # amax sets the scale to 2^-3
    x[3, 32:64] = -torch.linspace(0, 7.5, 32)             # saturation past 6
    x[4, 64:96] = 1e-38                                   # tiny values (subnormal side)
    x[5, 96:128] = torch.tensor([-0.1, 0.1] * 16) * 1e-3  # values rounding to zero keep their sign
    x[5, 96] = 1.0
    xb = x.to(torch.bfloat16)
    q, s = moe.quantize_mx4(handle, xb.cuda())
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp4_quantize(xb)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 384), (1536 * 2, 4096)])
def test_tile_order_is_the_stated_byte_permutation(handle, rows, cols):
    # Tile order of one matrix: the 128-row x 128-element block (t, kb) is 8 KB
    # at block t * (cols // 128) + kb, its rows 64 bytes apart. Of a gate/up
    # pair: 16 KB per block, gate rows 0-63, up rows 0-63, gate rows 64-127, up
    # rows 64-127. Stated here as reshapes / transposes of the row-major bytes.
    g = torch.Generator().manual_seed(rows)
    q0 = torch.randint(0, 256, (rows, cols // 2), dtype=torch.int32, generator=g).to(torch.uint8)
    q1 = torch.randint(0, 256, (rows, cols // 2), dtype=torch.int32, generator=g).to(torch.uint8)
    nt, nk = rows // 128, cols // 128
    t = moe.tile_mxfp4(handle, q0.cuda())
    tp = moe.tile_mxfp4(handle, q0.cuda(), q1.cuda())
    torch.cuda.synchronize()
    blocks0 = q0.numpy().reshape(nt, 128, nk, 64).transpose(0, 2, 1, 3)     # [t, kb, row, byte]
    assert np.array_equal(t.cpu().numpy().reshape(-1), blocks0.reshape(-1))
    halves0 = blocks0.reshape(nt, nk, 2, 64, 64)                            # [t, kb, half, row, byte]
    halves1 = q1.numpy().reshape(nt, 128, nk, 64).transpose(0, 2, 1, 3).reshape(nt, nk, 2, 64, 64)
    pair = np.stack([halves0, halves1], axis=3)                             # [t, kb, half, gate/up, row, byte]
    assert np.array_equal(tp.cpu().numpy().reshape(-1), pair.reshape(-1))


def _w4a8_weights_oracle(w):
    return {k: (oracle.mxfp4_quantize(v.cpu()) if k.startswith("w_") else oracle.mx_quantize(v.cpu()))
            for k, v in w.items()}


# MOE_OPT_MX_TILE: 0 automatic, 1 the 128-row tile, 2 the 256-row tile, 3 weights as M.
@pytest.mark.parametrize("tile", [0, 1, 2, 3])
@pytest.mark.parametrize("H,I,sizes", [(256, 128, [16, 0, 3, 1]), (512, 384, [0, 1, 37, 130, 300, 0])])
def test_w4a8_grouped_gemm_matches_oracle(handle, tile, H, I, sizes):
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(12)
    a = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    wg, wu, wd = ((torch.randn(*sh, generator=g) * 0.02).to(torch.bfloat16) for sh in ((G, I, H), (G, I, H), (G, H, I)))
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    mw = moe.quantize_weights_mx(handle, {"w_gate": wg.cuda(), "w_up": wu.cuda(), "w_down": wd.cuda()}, w4=True)
    assert mw["w_gate"].shape == (G, I, H // 2)
    pw = moe.pack_weights_mx(handle, mw)
    y = torch.full((rows, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.grouped_gemm_workspace_size(rows, H, I, moe.MOE_MXFP4_W4A8, num_groups=G), dtype=torch.uint8,
                     device="cuda")
    handle.set_option(moe.MOE_OPT_MX_TILE, tile)
    try:
        moe.grouped_swiglu_gemm(handle, aq, torch.from_numpy(offsets).cuda(), pw["w_gate"], pw["w_up"], pw["w_down"],
                                y, ws, num_groups=G, H=H, I=I, dtype=moe.MOE_MXFP4_W4A8, a_scale=as_,
                                s_gate=pw["s_gate"], s_down=pw["s_down"])
        torch.cuda.synchronize()
    finally:
        handle.set_option(moe.MOE_OPT_MX_TILE, 0)
    assert handle.device_status() == 0
    yh = y.cpu().numpy()
    xq, xs = oracle.mx_quantize(a)
    for gi in range(G):
        r0, r1 = offsets[gi], offsets[gi + 1]
        if r1 == r0:
            continue
        ref = oracle.swiglu_mlp_mx(xq[r0:r1], xs[r0:r1], oracle.mxfp4_quantize(wg[gi]), oracle.mxfp4_quantize(wu[gi]),
                                   oracle.mxfp4_quantize(wd[gi]), w4=True)
        _check(yh[r0:r1], ref, f"group {gi} tile {tile}")
    assert np.all(np.isnan(yh[offsets[-1]:]))


def _run_layer(shape, x, logits, w_bf16):
    layer = moe.MoELayer(shape, w_bf16, device=0)
    out = layer(x, logits)
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    return out


def test_w4a8_layer_tiny(handle):
    shape = synth.WORKLOADS["tiny"].with_(dtype="mxfp4")
    x, logits = synth.make_activations(shape, seed=0)
    w = synth.make_weights(shape, seed=0)
    out = _run_layer(shape, x.cuda(), logits.cuda(), {k: v.cuda() for k, v in w.items()})
    ref = oracle.layer_forward_mx(x, logits, _w4a8_weights_oracle(w), K=shape.K, scaling=shape.scaling, w4=True)
    _check(out.float().cpu().numpy(), ref, "tiny w4a8")


def test_w4a8_layer_ragged_shape(handle):
    shape = synth.MoEShape("w4r", T=45, H=384, E=13, K=3, I=256, I_shared=128, dtype="mxfp4")
    x, logits = synth.make_activations(shape, seed=5)
    w = synth.make_weights(shape, seed=5)
    out = _run_layer(shape, x.cuda(), logits.cuda(), {k: v.cuda() for k, v in w.items()})
    ref = oracle.layer_forward_mx(x, logits, _w4a8_weights_oracle(w), K=shape.K, scaling=shape.scaling, w4=True)
    _check(out.float().cpu().numpy(), ref, "ragged w4a8")


def test_w4a8_layer_full_size_tile_edges(handle):
    shape = synth.WORKLOADS["mxfp4"]
    x, logits = synth.make_activations(shape, device="cuda", seed=0)
    w = synth.make_weights(shape, device="cuda", seed=0)
    out = _run_layer(shape, x, logits, w)
    ridx, _ = oracle.route(logits.cpu().numpy(), shape.K, shape.scaling)
    tokens = edge_tokens(ridx, shape.E, sample=16, seed=4)
    ref = oracle.layer_forward_mx(x.cpu(), logits.cpu(), _w4a8_weights_oracle(w), K=shape.K, scaling=shape.scaling,
                                  tokens=tokens, w4=True)
    _check(out.float().cpu().numpy()[tokens], ref, "mxfp4 workload")


def test_w4a8_layer_decode_shape_all_tokens(handle):
    # The decode shape (T=64, E=192, K=8) with W4A8 routed experts: about three
    # rows per expert, so nearly every 128-row token tile is a partial one.
    shape = synth.WORKLOADS["decode"].with_(dtype="mxfp4")
    x, logits = synth.make_activations(shape, device="cuda", seed=3)
    w = synth.make_weights(shape, device="cuda", seed=3)
    out = _run_layer(shape, x, logits, w)
    ref = oracle.layer_forward_mx(x.cpu(), logits.cpu(), _w4a8_weights_oracle(w), K=shape.K, scaling=shape.scaling,
                                  w4=True)
    _check(out.float().cpu().numpy(), ref, "decode shape w4a8")
