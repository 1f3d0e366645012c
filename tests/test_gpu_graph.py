"""CUDA-graph capture of moe_layer_forward (the decode-style launch-bound
case): one captured call, side stream included, replays bit-identically to
eager calls on new inputs written into the captured buffers."""
import pytest
import torch

import routed_expert_ffn_04_gb300 as moe
import synth
from gpu_common import cfg_of

pytestmark = pytest.mark.gpu


def test_captured_layer_replays_like_eager():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    shape = synth.MoEShape("graph", T=64, H=1024, E=32, K=8, I=512, I_shared=512)
    handle = moe.Handle(0)
    cfg = cfg_of(shape)
    w = synth.make_weights(shape, device="cuda", seed=3)
    weights = moe.make_weights(w)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    x, logits = synth.make_activations(shape, device="cuda", seed=1)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):  # warm-up outside the graph
        moe.layer_forward(handle, cfg, weights, x, logits, out, ws, side=side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        moe.layer_forward(handle, cfg, weights, x, logits, out, ws, side=side)
    torch.cuda.synchronize()
    ref = torch.empty_like(out)
    for seed in (5, 6):
        x2, l2 = synth.make_activations(shape, device="cuda", seed=seed)
        moe.layer_forward(handle, cfg, weights, x2, l2, ref, ws, side=side)
        torch.cuda.synchronize()
        x.copy_(x2)
        logits.copy_(l2)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), seed
    assert handle.device_status() == 0
