"""Helpers shared by the GPU parity tests (not a test module).

Tolerances (fixed by the layer's specification for bf16 outputs):
  layer output vs the fp64 oracle: max-abs <= 2e-2 and relative L2 <= 1e-2.
Routing ids, expert counts and the permutation are compared bit-exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import routed_expert_ffn_04_gb300 as moe
import synth

MAX_ABS = 2e-2
REL_L2 = 1e-2
ROUTE_W_RTOL = 1e-5

WEIGHT_KEYS = ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down")


def cfg_of(shape, **kw):
    d = dict(T=shape.T, H=shape.H, E=shape.E, K=shape.K, I=shape.I, I_shared=shape.I_shared,
             scaling=shape.scaling, route_norm=shape.route_norm)
    d.update(kw)
    return moe.make_config(**d)


def make_problem(shape, seed=0, device="cpu"):
    """Seeded inputs; generated on `device` and also returned on cuda."""
    x, logits = synth.make_activations(shape, device=device, seed=seed)
    w = synth.make_weights(shape, device=device, seed=seed)
    dev = torch.device("cuda")
    return (x.to(dev), logits.to(dev), {k: v.to(dev) for k, v in w.items()})


def run_layer(handle, shape, x, logits, w, *, mode=0, side=True, scaling=None, out=None, fold=False):
    cfg = cfg_of(shape, **({} if scaling is None else {"scaling": scaling}))
    handle.set_option(moe.MOE_OPT_GEMM_MODE, mode)
    handle.set_option(moe.MOE_OPT_SHARED_FOLD, int(fold))
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    if out is None:
        out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device="cuda")
    side_stream = torch.cuda.Stream() if side else None
    moe.layer_forward(handle, cfg, moe.make_weights(w), x, logits, out, ws, side=side_stream)
    torch.cuda.synchronize()
    handle.set_option(moe.MOE_OPT_SHARED_FOLD, 0)
    assert handle.device_status() == 0
    return out


def oracle_layer(shape, x, logits, w, tokens=None, scaling=None):
    ws = [w.get(k) for k in WEIGHT_KEYS]
    if shape.I_shared == 0:
        ws[3:] = [None, None, None]
    out, idx, tw = oracle.layer_forward(x, logits.cpu(), *ws, K=shape.K,
                                        scaling=shape.scaling if scaling is None else scaling,
                                        route_norm=shape.route_norm, tokens=tokens)
    return out, idx, tw


def check_layer(out_gpu: torch.Tensor, ref: np.ndarray, rows=None, what=""):
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def sample_tokens(T, n, seed=0):
    rng = np.random.default_rng(seed)
    picks = set([0, T - 1]) | set(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(picks), np.int32)
