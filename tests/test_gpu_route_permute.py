"""GPU parity of routing (step 1) and the InitRouting permutation (step 2)
against the oracle: ids, counts, offsets, perm_src, flat_to_perm and the
gathered rows bit-exact; routing weights within 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import ROUTE_W_RTOL, cfg_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    return moe.Handle(0)


def _route(handle, shape, logits):
    cfg = cfg_of(shape)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    w = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    moe.route(handle, cfg, logits, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


ROUTE_CASES = {
    "tiny": synth.WORKLOADS["tiny"],
    "decode": synth.WORKLOADS["decode"],
    "prefill": synth.WORKLOADS["prefill"],
    "skewed": synth.WORKLOADS["skewed"],
    "e37_k5": synth.MoEShape("e37", T=333, H=64, E=37, K=5, I=64, I_shared=0),
    "e1024_k32": synth.MoEShape("max", T=100, H=64, E=1024, K=32, I=64, I_shared=0),
    "k_eq_e": synth.MoEShape("keqe", T=50, H=64, E=6, K=6, I=64, I_shared=0),
    "no_norm": synth.MoEShape("nonorm", T=64, H=64, E=64, K=4, I=64, I_shared=0, route_norm=False),
}


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_route_matches_oracle(handle, name):
    shape = ROUTE_CASES[name]
    _, logits = synth.make_activations(shape, device="cuda", seed=11)
    idx, w = _route(handle, shape, logits)
    ridx, rw = oracle.route(logits.cpu().numpy(), shape.K, shape.scaling, shape.route_norm)
    assert np.array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=ROUTE_W_RTOL, atol=0)


def test_route_ties_zeros_and_saturation(handle):
    shape = synth.MoEShape("ties", T=6, H=64, E=40, K=4, I=64, I_shared=0)
    rows = np.zeros((6, 40), np.float32)
    rows[0, :] = 0.5                     # all equal -> ids 0..3
    rows[1, :] = -3.0
    rows[1, [5, 9]] = [-0.0, 0.0]        # +-0 tie -> 5 then 9
    rows[2, :] = np.linspace(30, 31, 40)  # sigma saturates, logits still rank
    rows[3, :] = -1.0
    rows[3, [39, 33, 1]] = 2.0           # tie across lanes -> 1, 33, 39
    rows[4, :] = np.float32(-np.inf)
    rows[4, 7] = 1.0
    rows[5, :] = np.arange(40)[::-1]
    logits = torch.from_numpy(rows).cuda()
    idx, w = _route(handle, shape, logits)
    ridx, rw = oracle.route(rows, 4, shape.scaling)
    assert np.array_equal(idx, ridx)
    assert idx[0].tolist() == [0, 1, 2, 3] and idx[1, :2].tolist() == [5, 9] and idx[3, :3].tolist() == [1, 33, 39]
    finite = np.isfinite(rw)
    np.testing.assert_allclose(w[finite], rw[finite], rtol=ROUTE_W_RTOL)


def _permute(handle, shape, topk_idx, x):
    cfg = cfg_of(shape)
    TK = shape.T * shape.K
    dev = "cuda"
    counts = torch.empty(shape.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(shape.E + 1, dtype=torch.int32, device=dev)
    perm_src = torch.empty(max(TK, 1), dtype=torch.int32, device=dev)
    f2p = torch.empty(max(TK, 1), dtype=torch.int32, device=dev)
    x_perm = torch.empty((max(TK, 1), shape.H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(moe.permute_workspace_size(cfg), dtype=torch.uint8, device=dev)
    moe.permute(handle, cfg, x, topk_idx, counts, offsets, perm_src, f2p, x_perm, ws)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), offsets.cpu().numpy(), perm_src[:TK].cpu().numpy(), f2p[:TK].cpu().numpy(), x_perm[:TK]


PERM_CASES = {
    "tiny": synth.WORKLOADS["tiny"],
    "decode": synth.WORKLOADS["decode"],
    "prefill": synth.WORKLOADS["prefill"],
    "skewed": synth.WORKLOADS["skewed"],
    "ragged": synth.MoEShape("ragged", T=77, H=128, E=13, K=3, I=64, I_shared=0),
    "e1024": synth.MoEShape("e1024", T=300, H=64, E=1024, K=32, I=64, I_shared=0),
    "t1": synth.MoEShape("t1", T=1, H=64, E=8, K=2, I=64, I_shared=0),
    # one block up to 4096 pairs, a cluster of 8 blocks up to 262144, three kernels above
    "tk4096": synth.MoEShape("tk4096", T=512, H=64, E=192, K=8, I=64, I_shared=0),
    "tk4097": synth.MoEShape("tk4097", T=4097, H=64, E=37, K=1, I=64, I_shared=0),
    "tk16392": synth.MoEShape("tk16392", T=2049, H=64, E=192, K=8, I=64, I_shared=0),
    "tk262144": synth.MoEShape("tk262144", T=32768, H=64, E=256, K=8, I=64, I_shared=0),
    "tk262145": synth.MoEShape("tk262145", T=262145, H=64, E=64, K=1, I=64, I_shared=0),
    "e1024_cluster": synth.MoEShape("e1024c", T=3000, H=64, E=1024, K=8, I=64, I_shared=0),
    "e1024_one_block": synth.MoEShape("e1024s", T=200, H=64, E=1024, K=32, I=64, I_shared=0),
}


@pytest.mark.parametrize("name", list(PERM_CASES))
def test_permute_matches_oracle(handle, name):
    shape = PERM_CASES[name]
    x, logits = synth.make_activations(shape, device="cuda", seed=12)
    idx, _ = _route(handle, shape, logits)
    counts, offsets, perm_src, f2p, x_perm = _permute(handle, shape, torch.from_numpy(idx).cuda(), x)
    rc, ro, rp, rf = oracle.permute(idx, shape.E)
    assert np.array_equal(counts, rc)
    assert np.array_equal(offsets, ro)
    assert np.array_equal(perm_src, rp)
    assert np.array_equal(f2p, rf)
    # Gathered rows are bit copies of x[perm_src // K].
    ref_rows = x[torch.from_numpy(rp // shape.K).long().cuda()]
    assert torch.equal(x_perm.view(torch.int16), ref_rows.view(torch.int16))


def test_permute_all_tokens_on_one_expert(handle):
    shape = synth.MoEShape("hot", T=700, H=64, E=16, K=1, I=64, I_shared=0)
    idx = np.full((700, 1), 9, np.int32)
    x, _ = synth.make_activations(shape, device="cuda", seed=3)
    counts, offsets, perm_src, f2p, _ = _permute(handle, shape, torch.from_numpy(idx).cuda(), x)
    assert counts.tolist() == [0] * 9 + [700] + [0] * 6
    assert perm_src.tolist() == list(range(700))


def test_permute_zero_tokens(handle):
    shape = synth.MoEShape("empty", T=0, H=64, E=8, K=2, I=64, I_shared=0)
    x = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    counts, offsets, _, _, _ = _permute(handle, shape, idx, x)
    assert counts.tolist() == [0] * 8 and offsets.tolist() == [0] * 9


def test_bad_expert_id_is_reported(handle):
    shape = synth.MoEShape("bad", T=4, H=64, E=8, K=2, I=64, I_shared=0)
    idx = torch.tensor([[0, 1], [2, 99], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    handle.device_status()
    _permute(handle, shape, idx, x)
    assert handle.device_status() == 16  # MOE_DEV_BAD_EXPERT_ID
    assert handle.device_status() == 0   # cleared by the read


def test_combine_skips_dropped_pairs_silently(handle):
    # A pair with an expert id out of range is dropped by the permutation
    # (reported once there, flat_to_perm = -1). The combine then adds the
    # token's other slots only and reports nothing more.
    shape = synth.MoEShape("bad", T=4, H=64, E=8, K=2, I=64, I_shared=0)
    idx = torch.tensor([[0, 1], [2, 99], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    handle.device_status()
    _, _, _, f2p, _ = _permute(handle, shape, idx, x)
    assert handle.device_status() == 16  # MOE_DEV_BAD_EXPERT_ID, from the permutation
    assert f2p[3] == -1
    g = torch.Generator(device="cpu").manual_seed(5)
    y = torch.randn((shape.T * shape.K, shape.H), generator=g, dtype=torch.float32)
    w = torch.rand((shape.T, shape.K), generator=g, dtype=torch.float32)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    moe.combine(handle, cfg_of(shape), y.cuda(), w.cuda(), torch.from_numpy(f2p).cuda(), None, out)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    ref = np.zeros((shape.T, shape.H))
    for t in range(shape.T):
        for k in range(shape.K):
            p = f2p[t * shape.K + k]
            if p >= 0:
                ref[t] += float(w[t, k]) * y[p].double().numpy()
    got = out.float().cpu().numpy()
    # One bf16 rounding of an fp32 sum: within a bf16 half-ulp plus fp32 error.
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5)
