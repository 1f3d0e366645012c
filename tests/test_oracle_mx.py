"""Pins for the oracle's MXFP8 quantiser (E4M3 elements, E8M0 scale per 32).

The pages put the routed and shared Linears in W8A8 MXFP8 and quantise
activations dynamically ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战",
sections 8.2 and 六). The conversion rule is the OCP MX v1.0 one. The pins: the
E4M3 format table (golden fixture), torch's float8_e4m3fn conversion (a library
routine) on in-range values, exact round trips, zero blocks, saturation and the
rounding error bound.
"""
import numpy as np
import pytest
import torch

import oracle


def _points(golden_dir):
    pts = []
    for line in open(f"{golden_dir}/e4m3_points.txt"):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        pts.append((int(c, 16), float(v)))
    return pts


def test_e4m3_table_points(golden_dir):
    for code, v in _points(golden_dir):
        got = oracle.e4m3_value(code)
        assert got == v and np.signbit(got) == np.signbit(v), hex(code)
    assert np.isnan(oracle.e4m3_value(0x7F)) and np.isnan(oracle.e4m3_value(0xFF))
    vals = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))  # monotone magnitudes


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if np.isnan(ref[c]):
            assert np.isnan(v)
        else:
            assert v == ref[c], hex(c)


def test_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 0.05,
                        rng.standard_normal(2000) * 1e-3])
    # Midpoints between neighbouring codes exercise ties-to-even.
    mags = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (mags[:-1] + mags[1:]) / 2
    v = np.concatenate([v, mids, -mids]).astype(np.float32)  # midpoints are exact in fp32
    v = np.concatenate([v, np.array([-1e-4, 1e-4, -0.0, 0.0], np.float32)])  # round to +-0
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(a)) for a in v], np.uint8)
    assert np.array_equal(got, ref)


def test_saturation():
    assert oracle.e4m3_encode(460.0) == 0x7E
    assert oracle.e4m3_encode(511.9) == 0x7E
    assert oracle.e4m3_encode(-500.0) == 0xFE
    assert oracle.e4m3_encode(456.0) == 0x7E  # midpoint 448/464 -> even code 0x7E


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_block_scale_powers_of_two_and_zero_block():
    # Block 0: amax = 1.0 -> shared_exp = 0 - 8 -> E8M0 code 119; 1.0 / 2^-8 = 256 = code 0x78.
    # Block 1: all zero -> scale code 0, elements +0.
    # Block 2: amax = 2^5 exactly at a binade edge -> code 127 + 5 - 8.
    row = np.zeros(96, np.float32)
    row[0] = 1.0
    row[1] = -0.5
    row[64] = 32.0
    row[65] = 0.125
    q, s = oracle.mx_quantize(_bf16(row[None, :]))
    assert s[0].tolist() == [119, 0, 124]
    assert q[0, 0] == 0x78 and q[0, 1] == 0xF0  # -0.5/2^-8 = -128 = -(2^7)
    assert np.all(q[0, 32:64] == 0)
    deq = oracle.mx_dequantize(q, s)
    assert np.array_equal(deq[0], row.astype(np.float64))


def test_representable_values_round_trip_exactly():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 0x7F, size=(8, 64))
    signs = rng.choice([-1.0, 1.0], size=codes.shape)
    mags = np.vectorize(oracle.e4m3_value)(codes)
    base = (signs * mags)
    base[:, 0] = 448.0  # pin amax so the block scale is 2^(8-8) * 2^k below
    base[:, 32] = -448.0
    for k in (-3, 0, 4):
        v = base * 2.0 ** k
        q, s = oracle.mx_quantize(_bf16(v))
        # amax = 448 * 2^k -> floor(log2) = 8 + k -> shared exp k.
        assert np.all(s == 127 + k)
        assert np.array_equal(oracle.mx_dequantize(q, s), v.astype(np.float32).astype(np.float64))


def test_error_bound_random():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 128)) * np.exp(rng.uniform(-6, 6, (64, 1)))
    q, s = oracle.mx_quantize(v)
    deq = oracle.mx_dequantize(q, s)
    X = np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    r = np.abs(v) / X
    normal = (r >= 2.0 ** -6) & (r <= 448)
    err = np.abs(v - deq)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(v[normal]) * (1 + 1e-12))
    sub = r < 2.0 ** -6
    assert np.all(err[sub] <= X[sub] * 2.0 ** -10 * (1 + 1e-12))
    sat = r > 448
    assert np.all(np.abs(deq[sat]) == 448 * X[sat])
    # Every block's amax lands in [256, 512) before saturation.
    amax = np.abs(v).reshape(64, 4, 32).max(-1)
    ratio = amax / 2.0 ** (s.astype(np.float64) - 127)
    assert np.all((ratio >= 256) & (ratio < 512))


def test_mx_layer_close_to_bf16_layer_and_pins_scale_indexing():
    import synth

    sh = synth.WORKLOADS["tiny"]
    x, logits = synth.make_activations(sh, seed=3)
    w = synth.make_weights(sh, seed=3)
    mxw = {k: oracle.mx_quantize(v) for k, v in w.items()}
    out_mx = oracle.layer_forward_mx(x, logits, mxw, K=sh.K, scaling=sh.scaling)
    out_bf, _, _ = oracle.layer_forward(x, logits, *(w[k] for k in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")),
                                        K=sh.K, scaling=sh.scaling)
    rel = np.linalg.norm(out_mx - out_bf) / np.linalg.norm(out_bf)
    assert 1e-4 < rel < 0.08
    # Composition pin: the MX layer equals, per token, numpy matmuls over the
    # dequantised operands with h re-quantised by the (separately pinned) quantiser.
    deq = {k: oracle.mx_dequantize(*mxw[k]) for k in w}
    xd = oracle.mx_dequantize(*oracle.mx_quantize(x))
    _, idx, tw = oracle.layer_forward(x, logits, *(w[k] for k in ("w_gate", "w_up", "w_down")), K=sh.K,
                                      scaling=sh.scaling)

    def mlp(xrow, g_, u_, d_):
        g = g_ @ xrow
        u = u_ @ xrow
        h = g / (1.0 + np.exp(-g)) * u
        hq = oracle.mx_dequantize(*oracle.mx_quantize(h[None, :]))[0]
        return d_ @ hq

    ref = np.zeros_like(out_mx)
    for t in range(sh.T):
        ref[t] = mlp(xd[t], deq["ws_gate"], deq["ws_up"], deq["ws_down"])
        for k in range(sh.K):
            e = idx[t, k]
            ref[t] += tw[t, k] * mlp(xd[t], deq["w_gate"][e], deq["w_up"][e], deq["w_down"][e])
    np.testing.assert_allclose(out_mx, ref, rtol=1e-9, atol=1e-10)
    # Re-quantising an MX-dequantised tensor reproduces its codes and scales.
    wdq_up = _bf16(deq["w_up"].astype(np.float32))
    q2, s2 = oracle.mx_quantize(wdq_up)
    assert np.array_equal(q2, mxw["w_up"][0]) and np.array_equal(s2, mxw["w_up"][1])


def test_mx_mlp_on_quantised_rows_matches_numpy_composition():
    # Pins oracle.swiglu_mlp_mx: numpy matmuls over dequantised operands, with h
    # re-quantised by the (separately pinned) quantiser.
    g = torch.Generator().manual_seed(4)
    R, H, I = 9, 128, 96
    x = torch.randn(R, H, generator=g).to(torch.bfloat16)
    w = {k: (torch.randn(*sh, generator=g) * 0.05).to(torch.bfloat16)
         for k, sh in (("g", (I, H)), ("u", (I, H)), ("d", (H, I)))}
    xq, xs = oracle.mx_quantize(x)
    mw = {k: oracle.mx_quantize(v) for k, v in w.items()}
    y = oracle.swiglu_mlp_mx(xq, xs, mw["g"], mw["u"], mw["d"])
    xd = oracle.mx_dequantize(xq, xs)
    dg, du, dd = (oracle.mx_dequantize(*mw[k]) for k in ("g", "u", "d"))
    gg = xd @ dg.T
    h = gg / (1.0 + np.exp(-gg)) * (xd @ du.T)
    hq = oracle.mx_dequantize(*oracle.mx_quantize(h))
    np.testing.assert_allclose(y, hq @ dd.T, rtol=1e-9, atol=1e-12)
