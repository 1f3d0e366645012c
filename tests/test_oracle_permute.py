"""Pins for the oracle's InitRouting step (stable expert-contiguous permutation).

"腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the routed
path is InitRouting -> grouped GMM -> FinalizeRouting. The permutation is pinned
to numpy's stable argsort and bincount (library routines) and to the
bijection invariants.
"""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("T,K,E,seed", [(16, 2, 8, 0), (64, 8, 192, 1), (37, 3, 5, 2), (1, 4, 4, 3)])
def test_matches_numpy_stable_argsort(T, K, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm_src, flat_to_perm = oracle.permute(idx, E)
    flat = idx.ravel()
    assert np.array_equal(perm_src, np.argsort(flat, kind="stable"))
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts) and offsets[-1] == T * K
    assert np.array_equal(flat_to_perm[perm_src], np.arange(T * K))
    assert np.array_equal(np.sort(perm_src), np.arange(T * K))
    # Expert id non-decreasing along permuted rows; flat index ascending within an expert.
    ex = flat[perm_src]
    assert np.all(np.diff(ex) >= 0)
    for e in range(E):
        seg = perm_src[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_skewed_and_empty_experts():
    # All tokens on experts 2 and 5 of 8: the rest stay empty.
    idx = np.array([[5, 2]] * 10 + [[2, 5]] * 3, np.int32)
    counts, offsets, perm_src, _ = oracle.permute(idx, 8)
    assert counts.tolist() == [0, 0, 13, 0, 0, 13, 0, 0]
    assert offsets.tolist() == [0, 0, 0, 13, 13, 13, 26, 26, 26]
    # Expert 2 rows: flat indices of value 2 in ascending order.
    assert perm_src[:13].tolist() == [f for f in range(26) if idx.ravel()[f] == 2]


def test_zero_tokens():
    counts, offsets, perm_src, f2p = oracle.permute(np.zeros((0, 2), np.int32), 4)
    assert counts.tolist() == [0] * 4 and offsets.tolist() == [0] * 5 and perm_src.size == 0


def test_out_of_range_id_rejected():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 9]], np.int32), 4)
