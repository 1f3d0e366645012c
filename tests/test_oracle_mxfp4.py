"""Pins for the oracle's MXFP4 quantiser (E2M1 elements, E8M0 scale per 32)
and its W4A8 layer (MXFP4 routed-expert weights, MXFP8 activations, W8A8
shared expert: "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战",
section 8.2). The conversion rule is the OCP MX v1.0 one with E2M1's
emax_elem = 2. The pins: the E2M1 format table (golden fixture), encoding
against a brute-force nearest-value search with ties to even, exact round
trips, zero blocks, saturation, the scale rule, the nibble packing, and the
W4A8 layer against numpy matmuls over dequantised operands.
"""
import numpy as np
import torch

import oracle


def _points(golden_dir):
    pts = []
    for line in open(f"{golden_dir}/e2m1_points.txt"):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        pts.append((int(c, 16), float(v)))
    return pts


def test_e2m1_table(golden_dir):
    pts = _points(golden_dir)
    assert len(pts) == 16
    for code, v in pts:
        got = oracle.e2m1_value(code)
        assert got == v and np.signbit(got) == np.signbit(v), hex(code)


def test_encode_is_nearest_with_ties_to_even(golden_dir):
    # Brute force: the nearest of the 8 magnitudes; at an exact midpoint the one
    # whose code is even (mantissa bit 0); past 6 saturate.
    mags = np.array([v for c, v in _points(golden_dir) if c < 8])
    grid = np.concatenate([np.linspace(0, 7, 2801), mags, (mags[1:] + mags[:-1]) / 2])
    for a in grid:
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert oracle.e2m1_encode(a) == want, a
        assert oracle.e2m1_encode(-a) == (want | 8), -a
    # Named ties: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2.0, 3.5 -> 4.0, 5.0 -> 4.0.
    for a, code in ((0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (1e9, 7)):
        assert oracle.e2m1_encode(a) == code, a


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_block_rule_round_trip_zero_block_and_packing():
    # Block 0: the E2M1 grid times 2^-3 (amax 6 * 2^-3 -> shared exp -3); block 1: zeros
    # (scale 0, codes 0); block 2: the grid times 2^5 in reverse order.
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6] * 4, np.float64)
    row = np.concatenate([grid * 2.0 ** -3, np.zeros(32), grid[::-1] * 2.0 ** 5])
    q, s = oracle.mxfp4_quantize(_bf16(row[None, :]))
    assert q.shape == (1, 48) and s.shape == (1, 3)
    assert list(s[0]) == [127 - 3, 0, 127 + 5]
    assert np.all(q[0, 16:32] == 0)
    # Element 2j in the low nibble: codes 0,1 -> byte 0x10; 2,3 -> 0x32; ...
    assert list(q[0, :4]) == [0x10, 0x32, 0x54, 0x76]
    np.testing.assert_array_equal(oracle.mxfp4_dequantize(q, s)[0], row)


def test_saturation_and_scale_window():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((32, 128)) * np.exp(rng.uniform(-8, 8, (32, 1)))
    v = v.astype(np.float32).astype(np.float64)
    vb = _bf16(v)
    vq = vb.float().double().numpy()
    q, s = oracle.mxfp4_quantize(vb)
    deq = oracle.mxfp4_dequantize(q, s)
    X = np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    amax = np.abs(vq).reshape(32, 4, 32).max(-1)
    ratio = amax / 2.0 ** (s.astype(np.float64) - 127)
    assert np.all((ratio >= 4) & (ratio < 8))          # floor(log2 amax) - 2
    r = np.abs(vq) / X
    sat = r > 6
    assert np.all(np.abs(deq[sat]) == 6 * X[sat])
    # Below saturation the error is at most half the local spacing of the grid.
    spacing = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0)) * X
    assert np.all(np.abs(vq - deq)[~sat] <= spacing[~sat] / 2)


def test_w4a8_mlp_matches_numpy_composition():
    g = torch.Generator().manual_seed(6)
    R, H, I = 7, 128, 96
    x = torch.randn(R, H, generator=g).to(torch.bfloat16)
    w = {k: (torch.randn(*sh, generator=g) * 0.05).to(torch.bfloat16)
         for k, sh in (("g", (I, H)), ("u", (I, H)), ("d", (H, I)))}
    xq, xs = oracle.mx_quantize(x)
    mw = {k: oracle.mxfp4_quantize(v) for k, v in w.items()}
    y = oracle.swiglu_mlp_mx(xq, xs, mw["g"], mw["u"], mw["d"], w4=True)
    xd = oracle.mx_dequantize(xq, xs)
    dg, du, dd = (oracle.mxfp4_dequantize(*mw[k]) for k in ("g", "u", "d"))
    gg = xd @ dg.T
    h = gg / (1.0 + np.exp(-gg)) * (xd @ du.T)
    hq = oracle.mx_dequantize(*oracle.mx_quantize(h))
    np.testing.assert_allclose(y, hq @ dd.T, rtol=1e-9, atol=1e-12)


def test_w4a8_layer_composition_and_distance_to_bf16():
    import synth

    sh = synth.WORKLOADS["tiny"]
    x, logits = synth.make_activations(sh, seed=8)
    w = synth.make_weights(sh, seed=8)
    mw = {k: (oracle.mxfp4_quantize(v) if k.startswith("w_") else oracle.mx_quantize(v)) for k, v in w.items()}
    out = oracle.layer_forward_mx(x, logits, mw, K=sh.K, scaling=sh.scaling, w4=True)
    out_bf, idx, tw = oracle.layer_forward(x, logits, *(w[k] for k in ("w_gate", "w_up", "w_down", "ws_gate",
                                                                    "ws_up", "ws_down")), K=sh.K, scaling=sh.scaling)
    rel = np.linalg.norm(out - out_bf) / np.linalg.norm(out_bf)
    assert 0.02 < rel < 0.3   # 4-bit weights: well away from bf16, far from garbage
    deq = {k: (oracle.mxfp4_dequantize(*mw[k]) if k.startswith("w_") else oracle.mx_dequantize(*mw[k])) for k in w}
    xd = oracle.mx_dequantize(*oracle.mx_quantize(x))

    def mlp(xrow, g_, u_, d_):
        g = g_ @ xrow
        h = g / (1.0 + np.exp(-g)) * (u_ @ xrow)
        return d_ @ oracle.mx_dequantize(*oracle.mx_quantize(h[None, :]))[0]

    ref = np.zeros_like(out)
    for t in range(sh.T):
        ref[t] = mlp(xd[t], deq["ws_gate"], deq["ws_up"], deq["ws_down"])
        for k in range(sh.K):
            e = idx[t, k]
            ref[t] += tw[t, k] * mlp(xd[t], deq["w_gate"][e], deq["w_up"][e], deq["w_down"][e])
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-10)
