"""GPU parity of the MXFP8 path (E4M3 elements, E8M0 scale per 32 along K)
against the oracle's MX statement.

The quantiser and the MX permutation are integer/byte work and are compared
bit-exactly. The MX GEMM and layer are compared with the oracle's MX layer,
which quantises the bf16 weights with its own quantiser and computes in fp64.
The bar for MXFP8 outputs is relative L2 <= 3e-2. Because both sides use the
same quantised operands, the tests also check max-abs <= 2e-2, a tighter
diagnostic that a mis-indexed block scale would break.
"""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import cfg_of, edge_tokens

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
    return rel, err.max()


def test_quantiser_bit_exact(handle):
    g = torch.Generator().manual_seed(0)
    x = torch.randn(257, 512, generator=g) * torch.exp(torch.randn(257, 1, generator=g) * 3)
    x[0, :32] = 0.0                                # zero block -> scale 0, codes 0
    x[1, :32] = -0.0
    x[2, 32:64] = 1e-30                            # tiny values (fp32/bf16 subnormal side)
    x[3, :32] = torch.linspace(-3, 3, 32)
    x[3, 5] = 1000.0                               # outlier sets the block scale
    x[4, 64:96] = 2.0 ** 7                         # amax on a binade edge
    x[5, 96:128] = -448.0 * 2.0 ** -3
    xb = x.to(torch.bfloat16)
    q, s = moe.quantize_mx(handle, xb.cuda())
    torch.cuda.synchronize()
    rq, rs = oracle.mx_quantize(xb)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_weight_quantisation_matches_oracle(handle):
    shape = synth.WORKLOADS["tiny"]
    w = synth.make_weights(shape, seed=1)
    mx = moe.quantize_weights_mx(handle, {k: v.cuda() for k, v in w.items()})
    torch.cuda.synchronize()
    for k, v in w.items():
        rq, rs = oracle.mx_quantize(v)
        sk = ("ss_" + k[3:]) if k.startswith("ws_") else ("s_" + k[2:])
        assert np.array_equal(mx[k].cpu().numpy(), rq), k
        assert np.array_equal(mx[sk].cpu().numpy(), rs), k


@pytest.mark.parametrize("H", [256, 4096])
def test_mx_permute_gathers_codes_and_scales(handle, H):
    shape = synth.MoEShape("mxp", T=75, H=H, E=12, K=3, I=128, I_shared=0, dtype="mxfp8")
    x, logits = synth.make_activations(shape, device="cuda", seed=2)
    xq, xs = moe.quantize_mx(handle, x)
    cfg = cfg_of(shape)
    cfg.dtype = moe.MOE_MXFP8_E4M3
    TK = shape.T * shape.K
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    tw = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    moe.route(handle, cfg, logits, idx, tw)
    counts = torch.empty(shape.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(shape.E + 1, dtype=torch.int32, device="cuda")
    perm_src = torch.empty(TK, dtype=torch.int32, device="cuda")
    f2p = torch.empty(TK, dtype=torch.int32, device="cuda")
    xpq = torch.empty((TK, H), dtype=torch.uint8, device="cuda")
    xps = torch.empty((TK, H // 32), dtype=torch.uint8, device="cuda")
    ws = torch.empty(moe.permute_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    moe.permute(handle, cfg, xq, idx, counts, offsets, perm_src, f2p, xpq, ws, x_scale=xs, x_perm_scale=xps)
    torch.cuda.synchronize()
    rc, ro, rp, rf = oracle.permute(idx.cpu().numpy(), shape.E)
    assert np.array_equal(perm_src.cpu().numpy(), rp)
    src = torch.from_numpy(rp // shape.K).long().cuda()
    assert torch.equal(xpq, xq[src]) and torch.equal(xps, xs[src])


def _mx_weights_oracle(w):
    return {k: oracle.mx_quantize(v.cpu()) for k, v in w.items()}


def _atom_matrix(atoms, cols):
    """Inverse of the scale-atom layout (moe_pack_mx_scales in moe.h): row r of
    128-row block b, K-block j of atom (b, a) at byte 512 (b * cols/128 + a)
    + 16 (r % 32) + 4 (r / 32) + j. Returns the [rows, cols/32] matrix."""
    nk = cols // 128
    a = np.asarray(atoms, np.uint8).reshape(-1, nk, 32, 4, 4)   # [block, atom, r%32, r/32, j]
    a = a.transpose(0, 3, 2, 1, 4)                               # [block, r/32, r%32, atom, j]
    return a.reshape(-1, nk * 4)


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 512), (64 * 24, 4096)])
def test_pack_mx_scales_bit_exact(handle, rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    s0 = torch.randint(0, 255, (rows, cols // 32), generator=g, dtype=torch.uint8)
    s1 = torch.randint(0, 255, (rows, cols // 32), generator=g, dtype=torch.uint8)
    if rows % 128 == 0:
        got = _atom_matrix(moe.pack_mx_scales(handle, s0.cuda()).cpu().numpy(), cols)
        assert np.array_equal(got, s0.numpy())
    pair = _atom_matrix(moe.pack_mx_scales(handle, s0.cuda(), s1.cuda()).cpu().numpy(), cols)
    want = np.stack([s0.numpy().reshape(-1, 64, cols // 32), s1.numpy().reshape(-1, 64, cols // 32)], 1)
    assert np.array_equal(pair, want.reshape(2 * rows, cols // 32))


# MOE_OPT_MX_TILE: 0 automatic, 1 the 128-row tile, 2 the 256-row tile, 3 weights as M.
@pytest.mark.parametrize("tile", [0, 1, 2, 3])
@pytest.mark.parametrize("H,I,sizes", [(256, 128, [16, 0, 3, 1]), (512, 384, [0, 1, 37, 130, 300, 0])])
def test_mx_grouped_gemm_matches_oracle(handle, tile, H, I, sizes):
    G = len(sizes)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(3)
    a = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    wg, wu, wd = ((torch.randn(*sh, generator=g) * 0.02).to(torch.bfloat16) for sh in ((G, I, H), (G, I, H), (G, H, I)))
    aq, as_ = moe.quantize_mx(handle, a.cuda())
    mw = moe.quantize_weights_mx(handle, {"w_gate": wg.cuda(), "w_up": wu.cuda(), "w_down": wd.cuda()})
    pw = moe.pack_weights_mx(handle, mw)
    handle.set_option(moe.MOE_OPT_MX_TILE, tile)
    y = torch.full((rows, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.grouped_gemm_workspace_size(rows, H, I, moe.MOE_MXFP8_E4M3, num_groups=G), dtype=torch.uint8,
                     device="cuda")
    try:
        moe.grouped_swiglu_gemm(handle, aq, torch.from_numpy(offsets).cuda(), pw["w_gate"], pw["w_up"], pw["w_down"],
                                y, ws, num_groups=G, H=H, I=I, dtype=moe.MOE_MXFP8_E4M3, a_scale=as_,
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
        ref = oracle.swiglu_mlp_mx(xq[r0:r1], xs[r0:r1], oracle.mx_quantize(wg[gi]), oracle.mx_quantize(wu[gi]),
                                   oracle.mx_quantize(wd[gi]))
        _check(yh[r0:r1], ref, f"group {gi} tile {tile}")
    assert np.all(np.isnan(yh[offsets[-1]:]))


def _run_mx_layer(handle, shape, x, logits, w_bf16, mode=0):
    layer = moe.MoELayer(shape, w_bf16, device=0)
    layer.handle.set_option(moe.MOE_OPT_GEMM_MODE, mode)
    out = layer(x, logits)
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    return out


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_mx_layer_tiny(handle, mode):
    shape = synth.WORKLOADS["tiny"].with_(dtype="mxfp8")
    x, logits = synth.make_activations(shape, seed=0)
    w = synth.make_weights(shape, seed=0)
    out = _run_mx_layer(handle, shape, x.cuda(), logits.cuda(), {k: v.cuda() for k, v in w.items()}, mode)
    ref = oracle.layer_forward_mx(x, logits, _mx_weights_oracle(w), K=shape.K, scaling=shape.scaling)
    _check(out.float().cpu().numpy(), ref, f"tiny mx mode={mode}")


@pytest.mark.parametrize("mode", [1, 2])
def test_mx_layer_ragged_shape(handle, mode):
    shape = synth.MoEShape("mxr", T=45, H=384, E=13, K=3, I=256, I_shared=128, dtype="mxfp8")
    x, logits = synth.make_activations(shape, seed=5)
    w = synth.make_weights(shape, seed=5)
    out = _run_mx_layer(handle, shape, x.cuda(), logits.cuda(), {k: v.cuda() for k, v in w.items()}, mode)
    ref = oracle.layer_forward_mx(x, logits, _mx_weights_oracle(w), K=shape.K, scaling=shape.scaling)
    _check(out.float().cpu().numpy(), ref, f"ragged mx mode={mode}")


def test_mx_layer_full_size_tile_edges(handle):
    shape = synth.WORKLOADS["mxfp8"]
    x, logits = synth.make_activations(shape, device="cuda", seed=0)
    w = synth.make_weights(shape, device="cuda", seed=0)
    out = _run_mx_layer(handle, shape, x, logits, w)
    ridx, _ = oracle.route(logits.cpu().numpy(), shape.K, shape.scaling)
    tokens = edge_tokens(ridx, shape.E, sample=16, seed=2)
    ref = oracle.layer_forward_mx(x.cpu(), logits.cpu(), _mx_weights_oracle(w), K=shape.K, scaling=shape.scaling,
                                  tokens=tokens)
    _check(out.float().cpu().numpy()[tokens], ref, "mxfp8 workload")


@pytest.mark.parametrize("dtype", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("side", [True, False])
def test_prequantised_input_matches_bf16_input(handle, dtype, side):
    # moe_layer_forward with x already MXFP8 (codes + scales from
    # moe_quantize_mxfp8) gives the same bits as the layer that quantises the
    # bf16 x itself: the same codes and scales reach the same kernels.
    shape = synth.MoEShape("pre", T=300, H=512, E=24, K=4, I=256, I_shared=128, dtype=dtype)
    x, logits = synth.make_activations(shape, device="cuda", seed=9)
    w = synth.make_weights(shape, device="cuda", seed=9)
    layer = moe.MoELayer(shape, w, device=0, side_stream=side)
    a = layer(x, logits).clone()
    xq, xs = moe.quantize_mx(layer.handle, x)
    b = layer(xq, logits, x_scale=xs).clone()
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # And both match the MX oracle.
    if dtype == "mxfp4":  # routed weights MXFP4, shared W8A8
        wo = {k: (oracle.mxfp4_quantize(v.cpu()) if k.startswith("w_") else oracle.mx_quantize(v.cpu()))
              for k, v in w.items()}
    else:
        wo = _mx_weights_oracle(w)
    ref = oracle.layer_forward_mx(x.cpu(), logits.cpu(), wo, K=shape.K, scaling=shape.scaling, w4=dtype == "mxfp4")
    _check(b.float().cpu().numpy(), ref, f"pre-quantised {dtype}")
