"""GPU parity of the whole layer (moe_layer_forward) against the oracle.

Every workload shape is covered: tiny (all tokens), Hy3 decode (all 64
tokens), Hy3 prefill and the skewed Hy4-like load (sampled tokens at full
size, in the configuration the bench times), plus edge cases (one token,
ragged T, no shared expert, one expert, scaling 0) and invariants
(determinism, token-order equivariance, the side-stream join).

Tolerance: max-abs <= 2e-2 and relative L2 <= 1e-2 against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import (check_layer, check_layer_faithful, cfg_of, edge_tokens, make_problem, oracle_layer,
                        run_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    return moe.Handle(0)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("side", [True, False])
def test_tiny_all_tokens(handle, mode, side):
    shape = synth.WORKLOADS["tiny"]
    x, logits, w = make_problem(shape, seed=0)
    out = run_layer(handle, shape, x, logits, w, mode=mode, side=side)
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()})
    check_layer(out, ref, what=f"tiny mode={mode} side={side}")


@pytest.mark.parametrize("shape", [
    synth.MoEShape("t1", T=1, H=256, E=8, K=2, I=128, I_shared=128),
    synth.MoEShape("ragged", T=37, H=320, E=11, K=3, I=192, I_shared=64),
    synth.MoEShape("noshared", T=50, H=256, E=16, K=4, I=128, I_shared=0),
    synth.MoEShape("one_expert", T=40, H=256, E=1, K=1, I=256, I_shared=0, scaling=1.0),
    synth.MoEShape("wide", T=130, H=512, E=64, K=8, I=256, I_shared=256),
    # The limits: 1024 experts (1024 groups in the grouped GEMM's tile table), top-32.
    synth.MoEShape("e1024_k32", T=50, H=128, E=1024, K=32, I=128, I_shared=128),
], ids=lambda s: s.name)
@pytest.mark.parametrize("mode", [1, 2])
def test_edge_shapes(handle, shape, mode):
    x, logits, w = make_problem(shape, seed=4)
    out = run_layer(handle, shape, x, logits, w, mode=mode)
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()})
    check_layer(out, ref, what=f"{shape.name} mode={mode}")


def test_decode_all_tokens(handle):
    shape = synth.WORKLOADS["decode"]
    x, logits, w = make_problem(shape, seed=0, device="cuda")
    out = run_layer(handle, shape, x, logits, w)
    wc = {k: v.cpu() for k, v in w.items()}
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, wc)
    check_layer(out, ref, what="decode")
    # The other tiling agrees too.
    out2 = run_layer(handle, shape, x, logits, w, mode=2)
    check_layer(out2, ref, what="decode tokens-as-M")


@pytest.mark.parametrize("name", ["prefill", "skewed"])
def test_full_size_tile_edges(handle, name):
    # Every expert's first and last rows and its tile edges (edge_tokens), in
    # the launch configuration the bench times, plus random tokens.
    shape = synth.WORKLOADS[name]
    x, logits, w = make_problem(shape, seed=0, device="cuda")
    out = run_layer(handle, shape, x, logits, w)
    ridx, _ = oracle.route(logits.cpu().numpy(), shape.K, shape.scaling)
    tokens = edge_tokens(ridx, shape.E, sample=24, seed=1)
    wc = {k: v.cpu() for k, v in w.items()}
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, wc, tokens=tokens)
    check_layer(out, ref, rows=tokens, what=f"{name} ({len(tokens)} tokens)")


def test_prefill_all_tokens(handle):
    # All 8192 tokens (33.5M outputs) of the prefill workload against the
    # oracle: relative L2 over everything, and each output within 2e-2 or a
    # faithful bf16 rounding of the exact value (check_layer_faithful).
    shape = synth.WORKLOADS["prefill"]
    x, logits, w = make_problem(shape, seed=0, device="cuda")
    out = run_layer(handle, shape, x, logits, w)
    wc = {k: v.cpu() for k, v in w.items()}
    ref, _, _ = oracle_layer(shape, x.cpu(), logits, wc)
    n_far = check_layer_faithful(out, ref, what="prefill, every token")
    # A handful at most: the tail of the intermediate rounding's error.
    assert n_far <= 64, n_far


def test_scaling_zero_gives_shared_expert_exactly(handle):
    shape = synth.MoEShape("s0", T=33, H=256, E=8, K=2, I=128, I_shared=128)
    x, logits, w = make_problem(shape, seed=6)
    out = run_layer(handle, shape, x, logits, w, scaling=0.0)
    # The shared expert alone, through the grouped GEMM entry point (one group).
    y = torch.empty((shape.T, shape.H), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.grouped_gemm_workspace_size(shape.T, shape.H, shape.I_shared), dtype=torch.uint8, device="cuda")
    moe.grouped_swiglu_gemm(handle, x, None, w["ws_gate"], w["ws_up"], w["ws_down"], y, ws, num_groups=1,
                            H=shape.H, I=shape.I_shared)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), y.to(torch.bfloat16).view(torch.int16))


def test_deterministic_and_token_order_equivariant(handle):
    shape = synth.MoEShape("eq", T=96, H=512, E=32, K=4, I=256, I_shared=256)
    x, logits, w = make_problem(shape, seed=7)
    a = run_layer(handle, shape, x, logits, w).clone()
    b = run_layer(handle, shape, x, logits, w).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    p = torch.randperm(shape.T, generator=torch.Generator().manual_seed(1)).cuda()
    c = run_layer(handle, shape, x[p].contiguous(), logits[p].contiguous(), w)
    assert torch.equal(c.view(torch.int16), a[p].view(torch.int16))


def test_combine_forms_agree_bitwise(handle):
    # The combine splits H across blocks below 304 tokens and takes one block
    # per token from 304 up; the sum order is the same, and each row's GEMM
    # result does not depend on the tile it lands in, so the first 303 tokens
    # come out bit-identical either way.
    shape = synth.MoEShape("c304", T=304, H=256, E=16, K=4, I=128, I_shared=128)
    x, logits, w = make_problem(shape, seed=8)
    a = run_layer(handle, shape, x, logits, w).clone()
    small = shape.with_(T=303)
    b = run_layer(handle, small, x[:303].contiguous(), logits[:303].contiguous(), w)
    assert torch.equal(a[:303].view(torch.int16), b.view(torch.int16))
    ref, _, _ = oracle_layer(small, x[:303].cpu(), logits[:303], {k: v.cpu() for k, v in w.items()})
    check_layer(b, ref, what="303 tokens")


def test_side_stream_join_with_delayed_shared_expert(handle):
    # The side stream is held back by a bounded sleep before the call; the
    # main stream must still wait for the shared expert of THIS call.
    shape = synth.MoEShape("join", T=64, H=512, E=16, K=4, I=256, I_shared=512)
    x1, logits, w = make_problem(shape, seed=8)
    x2 = (x1.float() * -0.5).to(torch.bfloat16)
    cfg = cfg_of(shape)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    weights = moe.make_weights(w)
    handle.set_option(moe.MOE_OPT_GEMM_MODE, 0)
    moe.layer_forward(handle, cfg, weights, x1, logits, out, ws, side=side)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(50_000_000)  # tens of ms of spinning, then it returns
    moe.layer_forward(handle, cfg, weights, x2, logits, out, ws, side=side)
    torch.cuda.synchronize()
    ref, _, _ = oracle_layer(shape, x2.cpu(), logits, {k: v.cpu() for k, v in w.items()})
    check_layer(out, ref, what="delayed side stream")


def test_host_entry_point_matches_device_entry_point(handle):
    shape = synth.WORKLOADS["tiny"]
    x, logits, w = make_problem(shape, seed=9)
    dev_out = run_layer(handle, shape, x, logits, w).clone()
    cfg = cfg_of(shape)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    oh = torch.empty((shape.T, shape.H), dtype=torch.bfloat16).pin_memory()
    moe.layer_forward_host(handle, cfg, moe.make_weights(w), xh, lh, oh, ws, side=torch.cuda.Stream())
    assert torch.equal(oh.view(torch.int16), dev_out.cpu().view(torch.int16))


def test_bounded_wait_times_out_and_reports(handle):
    handle.device_status()
    handle.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 20_000)  # 20 ms
    try:
        handle.selftest_wait_timeout()
        torch.cuda.synchronize()
        assert handle.device_status() == moe.DEV_TIMEOUT_SELFTEST
        assert handle.device_status() == 0
        # The context is still usable afterwards.
        shape = synth.WORKLOADS["tiny"]
        x, logits, w = make_problem(shape, seed=0)
        handle.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 2_000_000)
        out = run_layer(handle, shape, x, logits, w)
        ref, _, _ = oracle_layer(shape, x.cpu(), logits, {k: v.cpu() for k, v in w.items()})
        check_layer(out, ref, what="after timeout")
    finally:
        handle.set_option(moe.MOE_OPT_WAIT_LIMIT_US, 2_000_000)


def test_shared_sm_split_does_not_change_the_result(handle):
    # MOE_OPT_SHARED_SMS only sizes the persistent grids of the two streams'
    # GEMMs; every row's arithmetic is the same, so the output is bit-identical.
    shape = synth.MoEShape("split", T=300, H=512, E=32, K=4, I=256, I_shared=256)
    x, logits, w = make_problem(shape, seed=11)
    outs = []
    for k in (0, 2, 3, 1000):
        handle.set_option(moe.MOE_OPT_SHARED_SMS, k)
        outs.append(run_layer(handle, shape, x, logits, w).clone())
    handle.set_option(moe.MOE_OPT_SHARED_SMS, 0)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    with pytest.raises(moe.MoEError):
        handle.set_option(moe.MOE_OPT_SHARED_SMS, -1)
