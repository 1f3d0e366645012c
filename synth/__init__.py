"""Seeded synthetic workloads for the MoE FFN layer.

This module only draws random inputs. It holds none of the layer's
arithmetic, and it is the one piece that both the CUDA-path tests and the
oracle-side tests use.

Workload shapes follow the pages' model facts:
  Hy3 ("腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战", section 一):
    hidden 4096, 192 routed experts, top-8, expert intermediate 1536,
    1 shared expert, router_scaling_factor 2.826, sigmoid routing, route_norm.
  Hy4 ("Hy4-preview（实验性）", section 1): 256 routed experts + 1 shared, top-8.

Distributions: x ~ N(0,1) (bf16), router logits ~ N(0,1) (fp32), weights
~ N(0, 0.02) (bf16, the 0.02 is a standard deviation). The skewed workload adds a
per-expert bias b_e ~ N(0, 2) (standard deviation 2) to every token's logits, so
some experts get no tokens and a few get many.

Every tensor comes from its own generator seeded with ``seed * 1000 + stream``
(x=1, logits=2, bias=3, w_gate=4, w_up=5, w_down=6, shared 7/8/9). A given
seed gives the same values on the same device type; CPU and CUDA draws differ.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch

SCALING_HY3 = 2.826


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    H: int
    E: int
    K: int
    I: int
    I_shared: int
    scaling: float = SCALING_HY3
    route_norm: bool = True
    dtype: str = "bf16"  # "bf16", "mxfp8" (W8A8) or "mxfp4" (W4A8: MXFP4 routed weights)
    skew: bool = False

    def as_dict(self):
        return asdict(self)

    def with_(self, **kw) -> "MoEShape":
        d = asdict(self)
        d.update(kw)
        return MoEShape(**d)


WORKLOADS = {
    # Small case the oracle finishes in well under a second.
    "tiny": MoEShape("tiny", T=16, H=256, E=8, K=2, I=128, I_shared=128),
    # Hy3 shape, decode (64 tokens).
    "decode": MoEShape("decode", T=64, H=4096, E=192, K=8, I=1536, I_shared=1536),
    # Hy3 shape, prefill (8192 tokens): near-uniform expert load.
    "prefill": MoEShape("prefill", T=8192, H=4096, E=192, K=8, I=1536, I_shared=1536),
    # Hy4-like expert count with a skewed load.
    "skewed": MoEShape("skewed", T=4096, H=4096, E=256, K=8, I=1536, I_shared=1536, skew=True),
    # Hy3 shape in MXFP8 (E4M3 + E8M0 per 32 along K).
    "mxfp8": MoEShape("mxfp8", T=2048, H=4096, E=192, K=8, I=1536, I_shared=1536, dtype="mxfp8"),
    # The same in W4A8: routed-expert weights MXFP4 (E2M1 + E8M0/32), MXFP8
    # activations, shared expert W8A8 ([Hy3] section 8.2).
    "mxfp4": MoEShape("mxfp4", T=2048, H=4096, E=192, K=8, I=1536, I_shared=1536, dtype="mxfp4"),
}

_STREAMS = dict(x=1, logits=2, bias=3, w_gate=4, w_up=5, w_down=6, ws_gate=7, ws_up=8, ws_down=9, w_router=10)


def _gen(device, seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _STREAMS[name])
    return g


def _normal(shape, std, dtype, device, seed, name):
    t = torch.empty(shape, dtype=dtype, device=device)
    t.normal_(0.0, std, generator=_gen(device, seed, name))
    return t


def make_activations(shape: MoEShape, device="cpu", seed: int = 0):
    """x [T,H] bf16 and router logits [T,E] fp32 for one layer call."""
    x = _normal((shape.T, shape.H), 1.0, torch.bfloat16, device, seed, "x")
    logits = _normal((shape.T, shape.E), 1.0, torch.float32, device, seed, "logits")
    if shape.skew:
        bias = _normal((shape.E,), 2.0, torch.float32, device, seed, "bias")
        logits = logits + bias[None, :]
    return x, logits


def make_router(shape: MoEShape, device="cpu", seed: int = 0, std: float = 0.02):
    """Router (gating projection) weights [E, H] bf16 ~ N(0, std), for the layer
    variant that computes the logits from x instead of taking them."""
    return _normal((shape.E, shape.H), std, torch.bfloat16, device, seed, "w_router")


def make_weights(shape: MoEShape, device="cpu", seed: int = 0, std: float = 0.02):
    """Routed experts: w_gate, w_up [E,I,H]; w_down [E,H,I]. Shared: ws_gate,
    ws_up [Is,H]; ws_down [H,Is]. All bf16, K-major (the reduction axis last)."""
    E, H, I, Is = shape.E, shape.H, shape.I, shape.I_shared
    w = {
        "w_gate": _normal((E, I, H), std, torch.bfloat16, device, seed, "w_gate"),
        "w_up": _normal((E, I, H), std, torch.bfloat16, device, seed, "w_up"),
        "w_down": _normal((E, H, I), std, torch.bfloat16, device, seed, "w_down"),
    }
    if Is > 0:
        w["ws_gate"] = _normal((Is, H), std, torch.bfloat16, device, seed, "ws_gate")
        w["ws_up"] = _normal((Is, H), std, torch.bfloat16, device, seed, "ws_up")
        w["ws_down"] = _normal((H, Is), std, torch.bfloat16, device, seed, "ws_down")
    return w
