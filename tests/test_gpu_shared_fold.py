"""GPU parity of the folded shared expert (MOE_OPT_SHARED_FOLD): the shared
MLP runs as one more group of the routed grouped GEMMs instead of on the side
stream ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 8.5: the
shared expert's output is added to the routed output; how it is scheduled does
not change the result). Same bars as the layer tests: max-abs <= 2e-2 and
relative L2 <= 1e-2 against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import check_layer, edge_tokens, make_problem, oracle_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    return moe.Handle(0)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_tiny_folded(handle, mode):
    shape = synth.WORKLOADS["tiny"]
    x, logits, w = make_problem(shape, seed=0)
    out = run_layer(handle, shape, x, logits, w, mode=mode, fold=True)
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()})
    check_layer(out, ref, what=f"tiny folded mode={mode}")


def test_decode_folded_all_tokens(handle):
    shape = synth.WORKLOADS["decode"]
    x, logits, w = make_problem(shape, seed=0, device="cuda")
    out = run_layer(handle, shape, x, logits, w, fold=True)
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()})
    check_layer(out, ref, what="decode folded")


def test_prefill_folded_tile_edges(handle):
    shape = synth.WORKLOADS["prefill"]
    x, logits, w = make_problem(shape, seed=0, device="cuda")
    out = run_layer(handle, shape, x, logits, w, fold=True)
    ridx, _ = oracle.route(logits.cpu().numpy(), shape.K, shape.scaling)
    tokens = edge_tokens(ridx, shape.E, sample=16, seed=3)
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()}, tokens=tokens)
    check_layer(out, ref, rows=tokens, what="prefill folded")


def test_fold_ignored_when_shapes_differ(handle):
    # I_shared != I: the option has no effect and the side stream runs the shared expert.
    shape = synth.MoEShape("ragged", T=37, H=320, E=11, K=3, I=192, I_shared=64)
    x, logits, w = make_problem(shape, seed=4)
    out = run_layer(handle, shape, x, logits, w, mode=2, fold=True)
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()})
    check_layer(out, ref, what="ragged, fold requested")


def test_folded_matches_side_stream(handle):
    shape = synth.MoEShape("eq", T=96, H=512, E=32, K=4, I=256, I_shared=256)
    x, logits, w = make_problem(shape, seed=9)
    a = run_layer(handle, shape, x, logits, w, mode=2).float()
    b = run_layer(handle, shape, x, logits, w, mode=2, fold=True).float()
    # One bf16 rounding apart at most (the same GEMM arithmetic, scheduled differently).
    diff = (a - b).abs().max().item()
    assert diff <= 2 ** -6 * max(1.0, a.abs().max().item()), diff
