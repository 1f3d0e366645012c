"""Host-side checks of the parity helpers' bf16 arithmetic (no GPU)."""
import numpy as np
import torch

from gpu_common import bf16_neighbours


def test_bf16_neighbours_enclose_and_contain_the_rounded_value():
    g = np.random.default_rng(3)
    ref = np.concatenate([g.normal(0, 3, 20000), [0.0, -0.0, 1.0, -4.0, 4.0625, 1e-30, -7.99]])
    lo, hi = bf16_neighbours(ref)
    # Both are bf16 numbers.
    for v in (lo, hi):
        t = torch.from_numpy(v.astype(np.float32))
        assert torch.equal(t.to(torch.bfloat16).float(), t)
    # They enclose the value (lo toward zero, hi away from it) ...
    assert np.all(np.abs(lo) <= np.abs(ref) + 1e-12) and np.all(np.abs(hi) >= np.abs(ref) - 1e-12)
    # ... at most one bf16 step apart (8 significant bits) ...
    step = np.abs(hi - lo)
    assert np.all(step <= np.abs(ref) * 2.0 ** -7 + 1e-300)
    # ... and round-to-nearest-even lands on one of them.
    rne = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.all((rne == lo) | (rne == hi))


def test_bf16_neighbours_of_a_representable_value_are_itself():
    v = np.array([4.03125, -0.5, 256.0])
    lo, hi = bf16_neighbours(v)
    assert np.array_equal(lo, v) and np.array_equal(hi, v)
