"""Pins of the oracle's gating projection, logits = x W_router^T in fp64
("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the main
stream runs gating before the routed path), against what the mathematics fixes
rather than a retyped formula:
  - one-hot router rows select columns of x exactly (catches a transposed
    operand or a wrong index);
  - a hand-computed example;
  - exact scaling by powers of two (linearity with no rounding);
  - sums of small integers, exact in fp64, at a size that spans many terms.
"""
import numpy as np
import torch

import oracle


def _bf16(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_one_hot_rows_select_columns():
    g = torch.Generator().manual_seed(3)
    T, H, E = 7, 64, 24
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    cols = [(5 * e + 3) % H for e in range(E)]  # distinct columns, not in order
    w = torch.zeros(E, H)
    for e, c in enumerate(cols):
        w[e, c] = 1.0
    got = oracle.gate(x, w.to(torch.bfloat16))
    assert got.shape == (T, E)
    np.testing.assert_array_equal(got, x.float().numpy().astype(np.float64)[:, cols])


def test_hand_computed_example():
    x = _bf16([[1.0, 2.0], [3.0, 4.0]])
    w = _bf16([[1.0, 0.0], [1.0, -1.0], [0.5, 0.25]])
    got = oracle.gate(x, w)
    np.testing.assert_array_equal(got, np.array([[1.0, -1.0, 1.0], [3.0, -1.0, 2.5]]))


def test_power_of_two_scaling_is_exact():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(5, 128, generator=g).to(torch.bfloat16)
    w = (torch.randn(9, 128, generator=g) * 0.02).to(torch.bfloat16)
    base = oracle.gate(x, w)
    np.testing.assert_array_equal(oracle.gate(x, (w.float() * 4.0).to(torch.bfloat16)), base * 4.0)
    np.testing.assert_array_equal(oracle.gate((x.float() * 0.5).to(torch.bfloat16), w), base * 0.5)


def test_integer_sums_are_exact():
    rng = np.random.default_rng(5)
    T, H, E = 4, 4096, 6
    x = rng.integers(-8, 9, size=(T, H)).astype(np.float32)
    w = rng.integers(-4, 5, size=(E, H)).astype(np.float32)
    want = x.astype(np.int64) @ w.astype(np.int64).T  # exact integer arithmetic
    got = oracle.gate(_bf16(x), _bf16(w))
    np.testing.assert_array_equal(got, want.astype(np.float64))
