"""CUDA-graph capture of moe_layer_forward and moe_layer_forward_gated (the
decode-style launch-bound case), in bf16, MXFP8 and W4A8: one captured call,
side stream included, replays bit-identically to eager calls on new inputs
written into the captured buffers."""
import pytest
import torch

import routed_expert_ffn_04_gb300 as moe
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,gated", [("bf16", False), ("bf16", True), ("mxfp8", False), ("mxfp4", False),
                                         ("mxfp8", True)])
def test_captured_layer_replays_like_eager(dtype, gated):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    shape = synth.MoEShape("graph", T=64, H=1024, E=32, K=8, I=512, I_shared=512, dtype=dtype)
    w = synth.make_weights(shape, device="cuda", seed=3)
    layer = moe.MoELayer(shape, w, device=0)  # MX: quantised and packed weights
    handle, cfg, weights, ws = layer.handle, layer.cfg, layer.weights, layer.ws
    w_router = synth.make_router(shape, device="cuda", seed=3) if gated else None
    x, logits = synth.make_activations(shape, device="cuda", seed=1)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()

    def call(dst, stream=None):
        if gated:
            moe.layer_forward_gated(handle, cfg, weights, w_router, x, dst, ws, main=stream, side=side)
        else:
            moe.layer_forward(handle, cfg, weights, x, logits, dst, ws, main=stream, side=side)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):  # warm-up outside the graph
        call(out, cap)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        call(out, cap)
    torch.cuda.synchronize()
    ref = torch.empty_like(out)
    for seed in (5, 6):
        x2, l2 = synth.make_activations(shape, device="cuda", seed=seed)
        x.copy_(x2)
        logits.copy_(l2)
        call(ref)  # eager, on the current stream
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), seed
    assert handle.device_status() == 0


def test_full_decode_workload_replays_like_eager():
    # The bench times graph replays of the full decode workload; eager calls
    # of that workload are checked against the oracle in test_gpu_layer.py.
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    moe.load(build_if_missing=True)
    shape = synth.WORKLOADS["decode"]
    layer = moe.MoELayer(shape, synth.make_weights(shape, device="cuda", seed=0), device=0)
    x, logits = synth.make_activations(shape, device="cuda", seed=0)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    ref = torch.empty_like(out)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        layer(x, logits, out, main=cap)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        layer(x, logits, out, main=cap)
    torch.cuda.synchronize()
    layer(x, logits, ref)
    torch.cuda.synchronize()
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert layer.handle.device_status() == 0
