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
    if err.size:
        i = np.unravel_index(int(err.argmax()), err.shape)
        small = np.abs(ref) < 8.0
        detail = (f" at ref={ref[i]:.5f} got={got[i]:.5f}; max |ref|={np.abs(ref).max():.3f}; "
                  f"max_abs where |ref|<8: {float(err[small].max()) if small.any() else 0.0:.3e}; "
                  f"n(err>2e-2)={int((err > MAX_ABS).sum())}")
    else:
        detail = ""
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}{detail}"
    return max_abs, rel


def bf16_neighbours(ref: np.ndarray):
    """The two bf16 values that enclose each fp64 value: toward zero and away
    from zero (equal to each other when the value is a bf16 number; the value
    is first taken to fp32, whose rounding is far below a bf16 step)."""
    r32 = np.ascontiguousarray(ref, np.float32)
    bits = r32.view(np.uint32)
    down = bits & np.uint32(0xFFFF0000)
    up = np.where(bits == down, down, down + np.uint32(0x10000))
    return down.view(np.float32).astype(np.float64), up.view(np.float32).astype(np.float64)


def check_layer_faithful(out_gpu: torch.Tensor, ref: np.ndarray, what=""):
    """Whole-output check for large workloads: relative L2 <= 1e-2, and every
    output within 2e-2 of the oracle or equal to one of the two bf16 numbers
    enclosing the oracle's value (a faithful rounding). Where |out| >= 4 the
    bf16 step is 1/32, so a computation error of a few 1e-3 (the bf16
    rounding of the GEMM-2 operand h) can move the fp32 sum across a rounding
    midpoint and the nearest bf16 value is then 0.016-0.031 away; the stated
    2e-2 bar is kept for every output it can hold for. Returns the count of
    outputs that needed the neighbour rule."""
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert rel <= REL_L2, f"{what}: rel_l2={rel:.3e}"
    err = np.abs(got - ref)
    far = err > MAX_ABS
    if far.any():
        lo, hi = bf16_neighbours(ref[far])
        g = got[far]
        ok = (g == lo) | (g == hi)
        assert ok.all(), (f"{what}: {int((~ok).sum())} outputs beyond 2e-2 and not a bf16 neighbour "
                          f"(worst {float(err[far][~ok].max()):.3e})")
    return int(far.sum())


def sample_tokens(T, n, seed=0):
    rng = np.random.default_rng(seed)
    picks = set([0, T - 1]) | set(rng.choice(T, size=min(n, T), replace=False).tolist())
    return np.array(sorted(picks), np.int32)


def edge_tokens(topk_idx, E, tile=128, block=32, sample=0, seed=0):
    """Tokens to check at full size: for every expert, the tokens whose
    permuted rows are the segment's first and last row, rows 127 and 128
    (the first tile edge of the tokens-as-M tiling), the first row of the last
    128-row tile and the row before it, and the first row of the last 32-row
    block (where the bulk-store epilogue of GEMM-2 hands over to row-by-row
    stores, and the 32-token tile edge of the weights-as-M tiling). Plus
    `sample` random tokens and the first and last token. The permutation is
    the oracle's, so the choice does not depend on the CUDA path."""
    idx = np.asarray(topk_idx)
    T, K = idx.shape
    counts, offsets, perm_src, _ = oracle.permute(idx, E)
    picks = set()
    for e in range(E):
        n = int(counts[e])
        if n == 0:
            continue
        last = (n - 1) // tile * tile
        for j in (0, n - 1, tile - 1, tile, last, last - 1, (n - 1) // block * block):
            if 0 <= j < n:
                picks.add(int(perm_src[offsets[e] + j]) // K)
    if sample:
        picks |= set(sample_tokens(T, sample, seed=seed).tolist())
    picks |= {0, T - 1}
    return np.array(sorted(picks), np.int32)
