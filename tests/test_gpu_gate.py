"""GPU checks of the gating projection fused with routing (moe_gate_route)
and of the layer that routes from it (moe_layer_forward_gated).

The router logits are bf16 products accumulated in fp32 (split-K on the
CUDA cores up to 256 tokens, tensor cores above), while the oracle computes
them in fp64, so two experts whose logits lie
within rounding of each other may legitimately be ordered either way. The
tests therefore check:
  - the logits against the oracle (|err| <= 2e-4 + 2e-4 |logit|);
  - the fused top-k against the standalone routing kernel on the same fp32
    logits, bit-exactly;
  - the chosen set against the oracle's logits: a valid top-K up to 1e-3;
  - the layer output against the oracle layer fed the oracle's logits, on
    the tokens routed the same way (max-abs 2e-2, rel-L2 1e-2).
"""
import numpy as np
import pytest
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import check_layer, cfg_of, edge_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def handle():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    return moe.Handle(0)


def _router(shape, seed=11):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape.E, shape.H, generator=g) * 0.02).to(torch.bfloat16)


# Up to 256 tokens (E <= 256) the split-K CUDA-core kernel runs, above that
# the tensor-core GEMM with the top-k in its epilogue; E > 256 writes the
# logits and runs the routing kernel.
GATE_SHAPES = [
    synth.WORKLOADS["decode"],                                                # split-K, 2 tokens a cluster
    synth.MoEShape("t1", T=1, H=4096, E=192, K=8, I=256, I_shared=0),         # one token
    synth.MoEShape("t5_h320", T=5, H=320, E=96, K=4, I=128, I_shared=0),      # K range not a multiple of 16
    synth.MoEShape("t100", T=100, H=1024, E=192, K=8, I=256, I_shared=0),     # 4 tokens a cluster
    synth.MoEShape("t256", T=256, H=1024, E=192, K=8, I=256, I_shared=0),     # largest split-K case
    synth.MoEShape("t257", T=257, H=1024, E=192, K=8, I=256, I_shared=0),     # smallest tensor-core case
    synth.MoEShape("t700_k12", T=700, H=512, E=96, K=12, I=256, I_shared=0),  # K > 8: K-round epilogue
    synth.MoEShape("prefill_like", T=1000, H=1024, E=192, K=8, I=256, I_shared=0),
    synth.MoEShape("e256", T=77, H=512, E=256, K=8, I=128, I_shared=0),       # ragged last cluster
    synth.MoEShape("e64k1", T=130, H=256, E=64, K=1, I=128, I_shared=0),      # four K pieces a CTA
    synth.MoEShape("e512", T=50, H=256, E=512, K=6, I=128, I_shared=0),       # logits + routing kernel path
]


@pytest.mark.parametrize("shape", GATE_SHAPES, ids=lambda s: s.name)
def test_gate_route(handle, shape):
    x, _ = synth.make_activations(shape, device="cuda", seed=3)
    wr = _router(shape).cuda()
    cfg = cfg_of(shape)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    w = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    logits = torch.empty((shape.T, shape.E), dtype=torch.float32, device="cuda")
    moe.gate_route(handle, cfg, x, wr, idx, w, logits_out=logits)
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    ref = oracle.gate(x.cpu(), wr.cpu())
    lg = logits.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lg - ref) <= 2e-4 + 2e-4 * np.abs(ref))
    # Fused top-k == the routing kernel on the same fp32 logits, bit for bit.
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    moe.route(handle, cfg, logits, idx2, w2)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    np.testing.assert_allclose(w.cpu().numpy(), w2.cpu().numpy(), rtol=1e-6, atol=0)
    # Valid top-K of the oracle logits up to near-ties.
    ids = idx.cpu().numpy()
    kth = -np.sort(-ref, axis=1)[:, shape.K - 1]
    chosen = np.take_along_axis(ref, ids, axis=1)
    assert np.all(chosen >= kth[:, None] - 1e-3)
    assert all(len(set(r)) == shape.K for r in ids.tolist())


@pytest.mark.parametrize("shape", [synth.WORKLOADS["decode"], GATE_SHAPES[5]], ids=lambda s: s.name)
def test_gate_route_without_logits_output(handle, shape):
    x, _ = synth.make_activations(shape, device="cuda", seed=4)
    wr = _router(shape).cuda()
    cfg = cfg_of(shape)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    w = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    moe.gate_route(handle, cfg, x, wr, idx, w)
    idx2, w2 = torch.empty_like(idx), torch.empty_like(w)
    moe.gate_route(handle, cfg, x, wr, idx2, w2, logits_out=torch.empty((shape.T, shape.E), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(w, w2)


@pytest.mark.parametrize("shape", [
    synth.WORKLOADS["tiny"], synth.WORKLOADS["decode"],
    synth.MoEShape("t600", T=600, H=512, E=64, K=4, I=128, I_shared=128),  # tensor-core gating
], ids=lambda s: s.name)
def test_gated_layer_matches_oracle(handle, shape):
    x, _ = synth.make_activations(shape, device="cuda", seed=5)
    w = synth.make_weights(shape, device="cuda", seed=5)
    wr = _router(shape, seed=12).cuda()
    cfg = cfg_of(shape)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    moe.layer_forward_gated(handle, cfg, moe.make_weights(w), wr, x, out, ws, side=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert handle.device_status() == 0
    ref_logits = oracle.gate(x.cpu(), wr.cpu()).astype(np.float32)
    wc = {k: v.cpu() for k, v in w.items()}
    ref, ridx, _ = oracle.layer_forward(x.cpu(), ref_logits, *(wc[k] for k in ("w_gate", "w_up", "w_down", "ws_gate",
                                                                                "ws_up", "ws_down")),
                                        K=shape.K, scaling=shape.scaling)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    tw = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    moe.gate_route(handle, cfg, x, wr, idx, tw)
    torch.cuda.synchronize()
    same = np.all(np.sort(idx.cpu().numpy(), 1) == np.sort(ridx, 1), axis=1)
    assert same.mean() > 0.9
    check_layer(out, ref[same], rows=np.nonzero(same)[0], what=f"gated {shape.name}")


@pytest.mark.parametrize("dtype", ["mxfp8", "mxfp4"])
def test_gated_mx_layer_matches_oracle(handle, dtype):
    # The router reads the bf16 x also in MX mode; the layer then quantises x
    # and runs the MX path on the routing the gating kernel chose.
    shape = synth.WORKLOADS["tiny"].with_(dtype=dtype, T=40)
    x, _ = synth.make_activations(shape, device="cuda", seed=6)
    w = synth.make_weights(shape, device="cuda", seed=6)
    wr = _router(shape, seed=13).cuda()
    layer = moe.MoELayer(shape, w, device=0)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    moe.layer_forward_gated(layer.handle, layer.cfg, layer.weights, wr, x, out, layer.ws, side=layer.side)
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    ref_logits = oracle.gate(x.cpu(), wr.cpu()).astype(np.float32)
    w4 = dtype == "mxfp4"
    mx_w = {k: (oracle.mxfp4_quantize(v.cpu()) if (w4 and k.startswith("w_")) else oracle.mx_quantize(v.cpu()))
            for k, v in w.items()}
    ref = oracle.layer_forward_mx(x.cpu(), ref_logits, mx_w, K=shape.K, scaling=shape.scaling, w4=w4)
    ridx, _ = oracle.route(ref_logits, shape.K, shape.scaling)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    tw = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    moe.gate_route(layer.handle, layer.cfg, x, wr, idx, tw)
    torch.cuda.synchronize()
    same = np.all(np.sort(idx.cpu().numpy(), 1) == np.sort(ridx, 1), axis=1)
    assert same.mean() > 0.9
    got = out.float().cpu().numpy().astype(np.float64)[same]
    r = ref[same]
    rel = np.linalg.norm(got - r) / np.linalg.norm(r)
    assert np.all(np.isfinite(got)) and rel <= 3e-2 and np.abs(got - r).max() <= 2e-2, (rel, np.abs(got - r).max())


def test_gated_full_prefill_tile_edges(handle):
    # The bench's gated prefill line: T = 8192 takes the tcgen05 gating path.
    shape = synth.WORKLOADS["prefill"]
    x, _ = synth.make_activations(shape, device="cuda", seed=0)
    w = synth.make_weights(shape, device="cuda", seed=0)
    wr = synth.make_router(shape, device="cuda", seed=0)
    layer = moe.MoELayer(shape, w, device=0)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    moe.layer_forward_gated(layer.handle, layer.cfg, layer.weights, wr, x, out, layer.ws, side=layer.side)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device="cuda")
    tw = torch.empty((shape.T, shape.K), dtype=torch.float32, device="cuda")
    moe.gate_route(layer.handle, layer.cfg, x, wr, idx, tw)
    torch.cuda.synchronize()
    assert layer.handle.device_status() == 0
    ref_logits = oracle.gate(x.cpu(), wr.cpu()).astype(np.float32)
    ridx, _ = oracle.route(ref_logits, shape.K, shape.scaling)
    tokens = edge_tokens(ridx, shape.E, sample=16, seed=3)
    same = np.all(np.sort(idx.cpu().numpy()[tokens], 1) == np.sort(ridx[tokens], 1), axis=1)
    assert same.mean() > 0.8
    tokens = tokens[same]
    wc = {k: v.cpu() for k, v in w.items()}
    ref, _, _ = oracle.layer_forward(x.cpu(), ref_logits, *(wc[k] for k in ("w_gate", "w_up", "w_down", "ws_gate",
                                                                             "ws_up", "ws_down")),
                                     K=shape.K, scaling=shape.scaling, tokens=tokens)
    check_layer(out, ref, rows=tokens, what="gated prefill")
