"""Pins for the oracle's routing step (sigmoid top-k, route_norm, scaling).

The routing follows "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战",
section 一: top-8 sigmoid routing over 192 experts, route_norm=True,
router_scaling_factor=2.826. Each check below pins the oracle to something
other than itself: brute force over all expert subsets, closed forms, and
the sorting routine of numpy.
"""
import itertools
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _facts(golden_dir):
    facts = {}
    for line in open(f"{golden_dir}/hy3_model_facts.txt"):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split()
        facts[k] = float(v)
    return facts


def test_workload_constants_match_pages(golden_dir):
    import synth

    f = _facts(golden_dir)
    d = synth.WORKLOADS["decode"]
    assert (d.H, d.E, d.K, d.I, d.I_shared) == (
        f["hy3.hidden_size"], f["hy3.n_routed_experts"], f["hy3.num_experts_per_tok"],
        f["hy3.moe_intermediate_size"], f["hy3.moe_intermediate_size"])
    assert d.scaling == f["hy3.router_scaling_factor"] and d.route_norm == bool(f["hy3.route_norm"])
    s = synth.WORKLOADS["skewed"]
    assert (s.E, s.K) == (f["hy4.n_routed_experts"], f["hy4.num_experts_per_tok"])


def test_topk_set_is_the_max_sum_subset_brute_force():
    # With distinct logits the top-K set is the unique K-subset of largest sum.
    rng = np.random.default_rng(1)
    T, E, K = 40, 8, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.route(logits, K, 1.0)
    for t in range(T):
        best = max(itertools.combinations(range(E), K), key=lambda s: sum(float(logits[t, j]) for j in s))
        assert set(idx[t].tolist()) == set(best)
        # Slot order: descending logit.
        vals = logits[t, idx[t]]
        assert np.all(np.diff(vals) < 0)


def test_full_order_when_k_equals_e_matches_numpy_lexsort():
    rng = np.random.default_rng(2)
    T, E = 25, 16
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 3] = logits[:, 7]  # planted ties
    idx, _ = oracle.route(logits, E, 1.0)
    for t in range(T):
        ref = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        assert idx[t].tolist() == ref.tolist()


@pytest.mark.parametrize(
    "row,K,expect",
    [
        ([0.5] * 6, 3, [0, 1, 2]),                      # all equal: lowest ids
        ([-0.0, 0.0, -1.0, -0.0], 2, [0, 1]),            # +0 and -0 tie
        ([30.0, 31.0, 30.0, -30.0], 3, [1, 0, 2]),       # sigma saturates in fp32; logits still rank
        ([1.0, 2.0, 2.0, 3.0, 2.0], 3, [3, 1, 2]),       # tie between ids 1, 2, 4 -> 1, 2
        ([-5.0, -4.0, -6.0], 1, [1]),
    ],
)
def test_ties_and_special_values(row, K, expect):
    idx, _ = oracle.route(np.array([row], np.float32), K, 1.0)
    assert idx[0].tolist() == expect


def test_closed_form_weights():
    # sigma(ln 3) = 3/4, sigma(0) = 1/2: route_norm weights 0.6 and 0.4, times scaling.
    s = 2.826
    row = np.array([[0.0, math.log(3.0), -5.0, -7.0]], np.float32)
    idx, w = oracle.route(row, 2, s)
    assert idx[0].tolist() == [1, 0]
    # ln 3 is rounded to fp32, hence the 1e-7 relative tolerance.
    assert w[0, 0] == pytest.approx(0.6 * s, rel=1e-7)
    assert w[0, 1] == pytest.approx(0.4 * s, rel=1e-7)
    # Without route_norm: w = scaling * sigma; sigma(0) = 1/2 exactly.
    idx, w = oracle.route(np.array([[0.0, -1.0]], np.float32), 1, s, route_norm=False)
    assert w[0, 0] == s / 2


def test_k1_weight_is_exactly_scaling_and_sums():
    rng = np.random.default_rng(3)
    logits = (rng.standard_normal((50, 12)) * 4).astype(np.float32)
    _, w1 = oracle.route(logits, 1, 2.826)
    assert np.all(w1 == 2.826)
    _, w = oracle.route(logits, 5, 2.826)
    assert np.allclose(w.sum(1), 2.826, rtol=0, atol=1e-12)
    _, w_unit = oracle.route(logits, 5, 1.0)
    assert np.allclose(w_unit.sum(1), 1.0, rtol=0, atol=1e-14)
    assert np.all(w > 0)


def test_rows_are_independent():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((30, 10)).astype(np.float32)
    idx, w = oracle.route(logits, 4, 2.826)
    for t in (0, 7, 29):
        i1, w1 = oracle.route(logits[t:t + 1], 4, 2.826)
        assert np.array_equal(i1[0], idx[t]) and np.array_equal(w1[0], w[t])


def test_weights_follow_logistic_function_closed_form():
    # Values of the logistic function at a few points (textbook closed forms):
    # sigma(0)=1/2; sigma(ln 2)=2/3; sigma(-ln 2)=1/3 -> route_norm of {ln2, 0, -ln2}
    # is (2/3, 1/2, 1/3) / (3/2) = (4/9, 1/3, 2/9).
    row = np.array([[math.log(2.0), 0.0, -math.log(2.0), -9.0]], np.float32)
    idx, w = oracle.route(row, 3, 1.0)
    assert idx[0].tolist() == [0, 1, 2]
    np.testing.assert_allclose(w[0], [4 / 9, 1 / 3, 2 / 9], rtol=1e-7)


def test_bad_sizes_rejected():
    with pytest.raises(ValueError):
        oracle.route(np.zeros((2, 3), np.float32), 4, 1.0)


def test_gate_matches_numpy_matmul():
    import torch

    g = torch.Generator().manual_seed(7)
    x = torch.randn(13, 96, generator=g).to(torch.bfloat16)
    w = (torch.randn(24, 96, generator=g) * 0.1).to(torch.bfloat16)
    ref = x.double().numpy() @ w.double().numpy().T
    np.testing.assert_allclose(oracle.gate(x, w), ref, rtol=1e-12, atol=1e-12)
    # A one-hot router row picks out one input column exactly.
    w1 = torch.zeros(4, 96, dtype=torch.bfloat16)
    w1[2, 17] = 1.0
    assert np.array_equal(oracle.gate(x, w1)[:, 2], x[:, 17].double().numpy())
