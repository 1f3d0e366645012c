#!/usr/bin/env python
"""Benchmark of the sigmoid-routed top-k MoE FFN layer (forward) on GB300.

One step = one whole layer call (routing, permutation, grouped SwiGLU GEMMs,
combine, shared expert on its own stream) on one batch of synthetic inputs
that are already resident in HBM. Default workload: the Hy3-shape decode
layer (T=64 tokens, H=4096, E=192 routed experts, top-8, I=1536, one shared
expert of I=1536, bf16 weights ~N(0, 0.02)).

Prints ONE JSON line (rank 0). Multi-GPU (torchrun): every rank runs its own
replica on its own tokens (no collective on the data path); `value` is the
tokens of all ranks divided by the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|skewed|mxfp8|mxfp4|tiny]
  python bench.py --impl reference ...   # the CPU oracle, timed on the host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MoE-layer tokens/sec at Hy3 shape; achieved HBM GB/s (decode) and TFLOP/s (prefill) vs peak")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the routed
# GEMM-1 launch, captured with ncu on a reduced-expert case of each workload
# (decode, MXFP8 and W4A8 at E = 48, prefill at E = 32; summarised in
# profiles/gemm1_traffic_reduced_e.md), as a ratio to that case's algorithmic
# GEMM-1 bytes. The full workload's traffic is reported as that ratio times
# its own algorithmic bytes (traffic grows with the bytes the launch must
# move: the touched experts' weights, the activation rows, h). A value is
# reported only while the GEMM sources still hash as they did for the capture.
# Per workload: the sources of its GEMM-1 kernel, their hash when captured, and
# the captured ratio of traffic to algorithmic bytes.
GEMM1_TRAFFIC = {
    "decode": (('gemm.cu', 'gemm_sched.cuh', 'ptx.cuh'), "5a8519b54d77f16e", (1212235264 + 3315200) / 1213726720),      # E = 48
    "prefill": (('gemm.cu', 'gemm_sched.cuh', 'ptx.cuh'), "5a8519b54d77f16e", (1164402432 + 191267840) / 1073741824),  # E = 32, A gathered
    "mxfp8": (('gemm_mx.cu', 'gemm_mx_wide.cu', 'gemm_sched.cuh', 'ptx.cuh'), "681f1db6bab86a2c", (693172736 + 23758848) / 718012416),  # E = 48, 256-row tile
    "mxfp4": (('gemm_mx.cu', 'gemm_mx_wide.cu', 'gemm_sched.cuh', 'ptx.cuh'), "681f1db6bab86a2c", (390695168 + 22090496) / 416022528),  # E = 48, 256-row tile
    # the decode shape with MX operands (--dtype): the weights-as-M GEMM-1
    "decode:mxfp8": (('gemm_mx_swap.cu', 'gemm_sched.cuh', 'ptx.cuh'), "76992db8f54232a1", (625859072 + 3213056) / 625827840),   # E = 48
    "decode:mxfp4": (('gemm_mx_swap.cu', 'gemm_sched.cuh', 'ptx.cuh'), "76992db8f54232a1", (323884032 + 2906112) / 323837952),   # E = 48
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=["tiny", "decode", "prefill", "skewed", "mxfp8", "mxfp4"])
    ap.add_argument("--dtype", default=None, choices=["bf16", "mxfp8", "mxfp4"],
                    help="the workload's shape with these operands (mxfp4: W4A8) instead of its own")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="with the default decode workload, skip the companion prefill measurement")
    ap.add_argument("--eager", action="store_true",
                    help="time eager layer calls; by default one captured call is replayed as a CUDA graph")
    ap.add_argument("--graph", action="store_true", help="(the default) time CUDA-graph replays")
    ap.add_argument("--gated", action="store_true",
                    help="compute the logits from router weights inside the layer (gating fused with routing)")
    ap.add_argument("--shared-fold", action="store_true",
                    help="run the shared expert as one more group of the routed GEMMs (bf16, I_shared == I)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-overlap", action="store_true",
                    help="skip the shared-expert overlap measurement (shorter runs, e.g. under a profiler)")
    ap.add_argument("--gemm-mode", type=int, default=0,
                    help="MOE_OPT_GEMM_MODE for the timed calls (0 automatic, 1 weights-as-M, 2 tokens-as-M, 3 CTA pair)")
    ap.add_argument("--mx-tile", type=int, default=0,
                    help="MOE_OPT_MX_TILE for the timed calls (0 automatic, 1 128-row, 2 256-row, 3 weights as M)")
    ap.add_argument("--ab-gemm-modes", default="",
                    help="comma-separated GEMM modes to time against each other (interleaved graph replays)")
    ap.add_argument("--ab-option", default="",
                    help="OPTION=v1,v2,...: time the layer with each value of a handle option (by number) "
                         "against each other, as --ab-gemm-modes does")
    ap.add_argument("--shared-sms-sweep", default="",
                    help="comma-separated MOE_OPT_SHARED_SMS values to add to the overlap measurement")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the routed expert count (smaller device footprint for profiler captures)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def dist_max(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, ms_local: float, world: int, device) -> tuple[float, float]:
    """Whole-job throughput: tokens of all ranks over the slowest rank's time."""
    ms = dist_max(ms_local, world, device)
    return tokens_per_rank * world / (ms * 1e-3), ms


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.lines = []

    def start(self):
        import torch

        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.device_index).uuid)
        except Exception:
            uuid = str(self.device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100", "-i", uuid],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "samples": len(sms),
                "reasons": sorted(reasons)}


def algorithmic_work(shape, counts, gated=False, gathered=False):
    """Bytes the layer must move and FLOPs it must do, from the expert counts.
    gathered: GEMM-1 reads its A rows from x itself (T rows) instead of from
    the permuted copy (T*K rows)."""
    H, I, Is, T, E, K = shape.H, shape.I, shape.I_shared, shape.T, shape.E, shape.K
    touched = int((counts > 0).sum())
    # Bytes per GEMM operand element: bf16, or an MX code (E4M3: 1 byte, E2M1:
    # half a byte) plus its share of the E8M0 scale (one per 32). W4A8 has E2M1
    # routed weights and E4M3 activations and shared weights. x, logits and out
    # are bf16 / fp32 either way.
    mx = shape.dtype in ("mxfp8", "mxfp4")
    ab = 1 + 1 / 32 if mx else 2                                  # activations, shared weights
    wb = 0.5 + 1 / 32 if shape.dtype == "mxfp4" else ab           # routed weights
    w_expert = 3 * H * I * wb
    w_shared = 3 * H * Is * ab
    # x, logits (or, gated, the [E, H] bf16 router weights) and out.
    layer_bytes = int(touched * w_expert + w_shared + T * H * 2 + (E * H * 2 if gated else T * E * 4) + T * H * 2)
    flops = 6 * H * I * T * K + 6 * H * Is * T + (2 * T * H * E if gated else 0)
    TK = T * K
    # GEMM-1 reads the touched experts' gate/up weights and x_perm (or, gathered,
    # x), and writes h.
    gemm1_bytes = int(touched * 2 * I * H * wb + (T if gathered else TK) * H * ab + TK * I * ab)
    return dict(touched=touched, layer_bytes=layer_bytes, flops=flops, gemm1_bytes=gemm1_bytes,
                gemm1_flops=4 * H * I * TK)


def oracle_layer_fn(shape, x, logits, w):
    """The oracle's statement of this workload's layer as f(tokens): bf16, or the
    MX layer on the oracle's own quantisation of the bf16 weights (W4A8: E2M1
    routed weights). Conversions happen here, outside any timing."""
    import oracle

    xb = oracle._bf16_bits(x.cpu())
    lh = np.ascontiguousarray(logits.cpu().numpy())
    keys = ["w_gate", "w_up", "w_down"] + (["ws_gate", "ws_up", "ws_down"] if shape.I_shared else [])
    if shape.dtype in ("mxfp8", "mxfp4"):
        w4 = shape.dtype == "mxfp4"
        mw = {k: (oracle.mxfp4_quantize(w[k].cpu()) if (w4 and k.startswith("w_")) else oracle.mx_quantize(w[k].cpu()))
              for k in keys}

        def run(toks):
            oracle.layer_forward_mx(xb, lh, mw, K=shape.K, scaling=shape.scaling, route_norm=shape.route_norm,
                                    tokens=toks, w4=w4)
        return run
    conv = [oracle._bf16_bits(w[k].cpu()) for k in keys]

    def run(toks):
        oracle.layer_forward(xb, lh, *conv, K=shape.K, scaling=shape.scaling, route_norm=shape.route_norm,
                             tokens=toks)
    return run


def cpu_oracle_rate(shape, x, logits, w, budget_s: float, max_tokens: int | None = None):
    """Time the oracle on a bounded sample of tokens; returns (tokens/s, n, seconds, threads)."""
    import oracle

    run = oracle_layer_fn(shape, x, logits, w)
    # Calibrate on a small batch (fixed per-call costs amortised), then size the sample.
    n_cal = min(shape.T, 16)
    t0 = time.perf_counter()
    run(np.arange(n_cal, dtype=np.int32))
    t1 = (time.perf_counter() - t0) / n_cal
    n = max(1, int(budget_s / max(t1, 1e-6)))
    if max_tokens is not None:
        n = min(n, max_tokens)
    toks = (np.arange(n) % shape.T).astype(np.int32)
    t0 = time.perf_counter()
    run(toks)
    dt = time.perf_counter() - t0
    return n / dt, n, dt, oracle.num_threads()


def source_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "routed_expert_ffn_04_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def time_graph(call, args, main, dev, world):
    """Capture one layer call (its side-stream fork and join included) as a
    CUDA graph and return the mean milliseconds of `args.steps` replays,
    between barriers and device synchronisations."""
    import torch

    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(main)
    with torch.cuda.stream(cap):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        call()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(main)
    for _ in range(args.steps):
        graph.replay()
    g1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    return g0.elapsed_time(g1) / args.steps


def measure_prefill(moe, synth, w, dev, main, peaks):
    """The metric's second half (TFLOP/s at prefill) measured in the same run
    as the decode line: the Hy3-shape prefill layer (T=8192) on the decode
    workload's weights (the same shapes and seed), CUDA-graph replays and
    stage-timed eager calls, with its own clock samples."""
    import types

    import torch

    shape = synth.WORKLOADS["prefill"]
    x, logits = synth.make_activations(shape, device=dev, seed=0)
    layer = moe.MoELayer(shape, w, device=dev.index)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device=dev)
    tw = torch.empty((shape.T, shape.K), dtype=torch.float32, device=dev)
    moe.route(layer.handle, layer.cfg, logits, idx, tw)
    counts = torch.bincount(idx.flatten().long(), minlength=shape.E).cpu().numpy()
    work = algorithmic_work(shape, counts, gathered=True)

    def call():
        layer(x, logits, out)

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    layer.handle.set_option(moe.MOE_OPT_STAGE_TIMING, 1)
    for _ in range(10):
        call()
    torch.cuda.synchronize()
    stage_ms, _ = layer.handle.stage_times()
    layer.handle.set_option(moe.MOE_OPT_STAGE_TIMING, 0)
    ms = time_graph(call, types.SimpleNamespace(steps=30, warmup=5), main, dev, 1)
    clocks = sampler.stop()
    if layer.handle.device_status() != 0:
        raise RuntimeError("device status set during the prefill measurement")
    sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    burst = float(peaks["bf16_tflops"])
    g1 = work["gemm1_flops"] / (stage_ms["gemm_gate_up"] * 1e-3) / 1e12
    lay = work["flops"] / (ms * 1e-3) / 1e12
    return {
        "workload": f"Hy3-shape prefill MoE layer (T={shape.T}) on the decode weights",
        "metric": "tokens/s; TFLOP/s vs the measured bf16 peaks (sustained, burst)",
        "value": round(shape.T / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "launch": "CUDA graph replay of one captured layer call (30 replays)",
        "layer_tflops": round(lay, 1), "layer_frac_sustained": round(lay / sustained, 4),
        "layer_frac_burst": round(lay / burst, 4),
        "gemm1_tflops": round(g1, 1), "gemm1_frac_sustained": round(g1 / sustained, 4),
        "gemm1_frac_burst": round(g1 / burst, 4),
        "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
        "clocks": clocks,
    }


def _spread(ms):
    a = np.asarray(ms)
    return {"median": round(float(np.median(a)), 5), "p10": round(float(np.percentile(a, 10)), 5),
            "p90": round(float(np.percentile(a, 90)), 5)}


def interleaved_replays(variants, main, dev, rounds=200):
    """Capture one CUDA graph per variant (name -> (setup, call); setup runs
    before the capture, e.g. to set a handle option baked into the launches)
    and time their replays interleaved round by round, the first of each
    round rotating; returns name -> list of ms."""
    import torch

    graphs = {}
    for name, (setup, fn) in variants.items():
        setup()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(main)
        with torch.cuda.stream(cap):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        torch.cuda.synchronize()
        graphs[name] = g
    names = list(graphs)
    times = {n: [] for n in names}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for r in range(rounds + 5):
        order = names[r % len(names):] + names[:r % len(names)]
        for n in order:
            e0.record(main)
            graphs[n].replay()
            e1.record(main)
            torch.cuda.synchronize()
            if r >= 5:
                times[n].append(e0.elapsed_time(e1))
    return times


def measure_gemm_modes(moe, layer, modes, call, main, dev, rounds=200, option=None, restore=0):
    """The layer with each value of a handle option (default: the grouped-GEMM
    tiling): interleaved graph replays, and per-stage device times from 30
    eager calls each."""
    import torch

    opt = moe.MOE_OPT_GEMM_MODE if option is None else option

    def setter(m):
        return lambda: layer.handle.set_option(opt, m)

    times = interleaved_replays({f"mode{m}": (setter(m), call) for m in modes}, main, dev, rounds)
    stages = {}
    for m in modes:
        layer.handle.set_option(opt, m)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        layer.handle.set_option(moe.MOE_OPT_STAGE_TIMING, 1)
        for _ in range(30):
            call()
        torch.cuda.synchronize()
        st, _ = layer.handle.stage_times()
        layer.handle.set_option(moe.MOE_OPT_STAGE_TIMING, 0)
        stages[f"mode{m}"] = {k: round(v, 5) for k, v in st.items()}
    layer.handle.set_option(opt, restore)
    return {"option": opt,
            "method": f"graph replays, {rounds} interleaved rounds; stages from 30 eager calls",
            "ms": {n: _spread(v) for n, v in times.items()}, "stage_ms": stages}


def measure_overlap(moe, layer, shape, cfg, x, logits, w_router, out, main, dev, args, rounds=200):
    """Shared-expert overlap from interleaved graph replays (see run_ours), and
    an eager A/B of the side stream at normal and at high priority."""
    import torch

    cfg_none = moe.make_config(shape.T, shape.H, shape.E, shape.K, shape.I, 0, shape.scaling, shape.route_norm,
                               cfg.dtype)
    side_hi = torch.cuda.Stream(device=dev, priority=-1)  # torch's high priority

    def fwd(c, side):
        if args.gated:
            moe.layer_forward_gated(layer.handle, c, layer.weights, w_router, x, out, layer.ws, side=side)
        else:
            moe.layer_forward(layer.handle, c, layer.weights, x, logits, out, layer.ws, side=side)

    calls = {"two_stream": lambda: fwd(cfg, layer.side), "serial": lambda: fwd(cfg, None),
             "no_shared": lambda: fwd(cfg_none, None)}
    sms = {}
    for v in filter(None, args.shared_sms_sweep.split(",")):
        calls[f"two_stream_sms{int(v)}"] = calls["two_stream"]
        sms[f"two_stream_sms{int(v)}"] = int(v)
    def sms_setter(k):  # the SM split between the streams is baked into the captured grids
        return lambda: layer.handle.set_option(moe.MOE_OPT_SHARED_SMS, k)

    times = interleaved_replays({n: (sms_setter(sms.get(n, 0)), fn) for n, fn in calls.items()}, main, dev, rounds)
    layer.handle.set_option(moe.MOE_OPT_SHARED_SMS, 0)
    names = list(times)
    med = {n: float(np.median(times[n])) for n in names}
    alone = med["serial"] - med["no_shared"]
    res = {"method": f"graph replays, {rounds} interleaved rounds, stage timing off",
           "ms": {n: _spread(times[n]) for n in names},
           "shared_alone_ms": round(alone, 5),
           "hidden_fraction": round((med["serial"] - med["two_stream"]) / alone, 3) if alone > 0 else None}
    # Eager calls: the side stream at normal and at high priority, interleaved.
    ev = {k: [] for k in ("normal", "high")}
    pairs = {"normal": layer.side, "high": side_hi}
    for r in range(rounds + 5):
        for k in (("normal", "high") if r % 2 == 0 else ("high", "normal")):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            fwd(cfg, pairs[k])
            e1.record(main)
            torch.cuda.synchronize()
            if r >= 5:
                ev[k].append(e0.elapsed_time(e1))
    res["eager_side_priority_ms"] = {k: _spread(v) for k, v in ev.items()}
    return res


def run_ours(args):
    import numpy as np
    import torch

    import routed_expert_ffn_04_gb300 as moe
    import synth

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape = synth.WORKLOADS[args.workload]
    if args.experts:
        shape = shape.with_(E=args.experts)
    if args.dtype:
        shape = shape.with_(dtype=args.dtype)
    moe.load()  # fails loudly when the library is not built

    x, logits = synth.make_activations(shape, device=dev, seed=rank)
    w = synth.make_weights(shape, device=dev, seed=0)
    layer = moe.MoELayer(shape, w, device=local)
    layer.handle.set_option(moe.MOE_OPT_GEMM_MODE, args.gemm_mode)
    layer.handle.set_option(moe.MOE_OPT_MX_TILE, args.mx_tile)
    if args.shared_fold:
        layer.handle.set_option(moe.MOE_OPT_SHARED_FOLD, 1)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    main = torch.cuda.current_stream(dev)

    # Routing counts of this input (for the algorithmic bytes), outside timing.
    cfg = layer.cfg
    idx = torch.empty((shape.T, shape.K), dtype=torch.int32, device=dev)
    tw = torch.empty((shape.T, shape.K), dtype=torch.float32, device=dev)
    w_router = synth.make_router(shape, device=dev, seed=0) if args.gated else None
    if args.gated:
        moe.gate_route(layer.handle, cfg, x, w_router, idx, tw)
    else:
        moe.route(layer.handle, cfg, logits, idx, tw)
    counts = torch.bincount(idx.flatten().long(), minlength=shape.E).cpu().numpy()
    # The layer's default path: bf16 GEMM-1 takes the tokens-as-M tiling above
    # 48 rows per expert on average, and then gathers its A rows from x.
    gathered = (shape.dtype == "bf16" and not args.shared_fold and args.gemm_mode in (0, 2)
                and (args.gemm_mode == 2 or shape.T * shape.K > 48 * shape.E))
    work = algorithmic_work(shape, counts, gated=args.gated, gathered=gathered)

    def call():
        if args.gated:
            moe.layer_forward_gated(layer.handle, cfg, layer.weights, w_router, x, out, layer.ws, side=layer.side)
        else:
            layer(x, logits, out)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    layer.handle.set_option(moe.MOE_OPT_STAGE_TIMING, 1)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(main)
    for _ in range(args.steps):
        call()
    ev1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    eager_ms = ev0.elapsed_time(ev1) / args.steps
    stage_ms, n_calls = layer.handle.stage_times()
    layer.handle.set_option(moe.MOE_OPT_STAGE_TIMING, 0)
    launch = "eager layer calls"
    graph_ms = None
    if not args.eager:
        try:
            graph_ms = time_graph(call, args, main, dev, world)
            launch = "CUDA graph replay of one captured layer call"
        except RuntimeError as exc:  # keep the eager number, say why
            launch = f"eager layer calls (graph capture failed: {str(exc).splitlines()[0][:120]})"
    value, ms = aggregate(shape.T, graph_ms if graph_ms is not None else eager_ms, world, dev)
    clocks = sampler.stop() if sampler else None  # sampled over every timed region
    status = layer.handle.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed region")

    # End-to-end through the public API: pinned host x (and logits) in, out back.
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    oh = torch.empty((shape.T, shape.H), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(1, min(args.e2e_steps, args.steps))

    def call_host():
        if args.gated:  # host x -> device, the gated layer, out -> host
            x.copy_(xh, non_blocking=True)
            moe.layer_forward_gated(layer.handle, cfg, layer.weights, w_router, x, out, layer.ws, side=layer.side)
            oh.copy_(out, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
        else:
            moe.layer_forward_host(layer.handle, cfg, layer.weights, xh, lh, oh, layer.ws, side=layer.side)

    for _ in range(3):
        call_host()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        call_host()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_ms = dist_max(e2e_ms, world, dev)

    # How much of the shared expert the second stream hides (the two-stream
    # timeline check, measured rather than assumed): graph replays of three
    # captured calls, interleaved round by round with stage timing off --
    # the two-stream layer, the same layer with the shared expert serial on
    # the main stream, and the layer without a shared expert. The shared MLP
    # alone costs serial - none; the second stream hides (serial - two) of it.
    overlap = None
    if shape.I_shared and not args.no_overlap and not (args.shared_fold and shape.dtype == "bf16"):
        overlap = measure_overlap(moe, layer, shape, cfg, x, logits, w_router, out, main, dev, args)

    gemm_ab = None
    if args.ab_gemm_modes:
        gemm_ab = measure_gemm_modes(moe, layer, [int(v) for v in args.ab_gemm_modes.split(",")], call, main, dev)
        layer.handle.set_option(moe.MOE_OPT_GEMM_MODE, args.gemm_mode)
    option_ab = None
    if args.ab_option:
        name, vals = args.ab_option.split("=")
        option_ab = measure_gemm_modes(moe, layer, [int(v) for v in vals.split(",")], call, main, dev,
                                       option=int(name), restore=int(vals.split(",")[-1]))

    peaks, peak_src = load_peaks()
    g1_ms = stage_ms["gemm_gate_up"]
    bound = "hbm" if args.workload in ("decode", "tiny", "mxfp8", "mxfp4") else "tensor"
    if bound == "hbm":
        achieved = work["gemm1_bytes"] / (g1_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        unit = "GB/s"
    else:
        achieved = work["gemm1_flops"] / (g1_ms * 1e-3) / 1e12
        peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
        if shape.dtype != "bf16":  # MX operands run at the fp8 rate: the measured bf16 peak x 2 (nominal ratio)
            peak *= 2.0
            peak_src += " x 2 (fp8 / bf16 nominal ratio)"
        unit = "TFLOP/s"
    traffic = None
    tkey = f"{args.workload}:{args.dtype}" if args.dtype else args.workload
    if (tkey in GEMM1_TRAFFIC and not args.experts and not args.gated
            and not args.shared_fold and args.gemm_mode == 0 and args.mx_tile == 0
            and source_sha(GEMM1_TRAFFIC[tkey][0]) == GEMM1_TRAFFIC[tkey][1]):
        traffic = int(round(GEMM1_TRAFFIC[tkey][2] * work["gemm1_bytes"]))
    layer_gbs = work["layer_bytes"] / (ms * 1e-3) / 1e9
    layer_tflops = work["flops"] / (ms * 1e-3) / 1e12
    # route 1; permute 1 (one block up to 16384 pairs, else 3) + row gather 1;
    # GEMMs 2; shared GEMMs 2 (folded: one small kernel that sets the extra
    # group's end); combine 1. MX adds the quantiser of x and the gather of
    # its scale atoms.
    tk = shape.T * shape.K
    permute_launches = (1 if tk <= 16384 else 3) + 1
    shared_launches = (1 if args.shared_fold and shape.dtype == "bf16" else 2) if shape.I_shared else 0
    launches_per_step = 1 + permute_launches + 2 + shared_launches + 1 + (2 if shape.dtype != "bf16" else 0)

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"mxfp8": "mxfp8 (E4M3 activations and weights, E8M0 scale per 32 along K, block-scaled "
                           "tensor cores, fp32 accumulate)",
                  "mxfp4": "w4a8 (E2M1 routed-expert weights, E4M3 activations and shared weights, E8M0 "
                           "scale per 32 along K, block-scaled tensor cores, fp32 accumulate)"}.get(shape.dtype,
                                                                                                    "bf16"),
        "data": "synthetic (seeded: x~N(0,1), logits~N(0,1), weights~N(0,0.02) bf16, random init)",
        "config": {
            "workload": (f"Hy3-shape {args.workload} MoE layer" if args.workload != "tiny" else "tiny MoE layer")
                        + (f" with E={shape.E}" if args.experts else "")
                        + (f", {args.dtype} operands" if args.dtype else ""),
            "T": shape.T, "H": shape.H, "E": shape.E, "K": shape.K, "I": shape.I, "I_shared": shape.I_shared,
            "scaling": shape.scaling, "route_norm": shape.route_norm, "skewed_logits": shape.skew,
            "l2": f"inputs larger than L2: {work['layer_bytes'] / 1e9:.2f} GB of weights+activations per step",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "launch": launch,
            "eager_ms_per_step": round(eager_ms, 5),
            "routing_input": ("router weights: gating kernel with the top-k fused in" if args.gated
                              else "given fp32 logits"),
            "shared_expert": ("one more group of the routed GEMMs" if args.shared_fold and shape.dtype == "bf16"
                              and shape.I_shared == shape.I else "side stream, event-ordered"),
            **({"mx_tile": args.mx_tile} if args.mx_tile else {}),
        },
        "roofline": {
            "kernel": "routed grouped GEMM-1 (gate/up + SwiGLU)",
            "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes": work["gemm1_bytes"], "avg_launch_ms": round(g1_ms, 5),
            "peak_source": f"{peak_src} ({'hbm_gbs' if bound == 'hbm' else 'bf16_tflops_sustained'})",
            "launches_timed": n_calls,
        },
        "layer": {
            "touched_experts": work["touched"], "algorithmic_bytes": work["layer_bytes"], "flops": work["flops"],
            "achieved_gbs": round(layer_gbs, 1), "hbm_frac": round(layer_gbs / float(peaks["hbm_gbs"]), 4),
            "achieved_tflops": round(layer_tflops, 2),
            "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
        },
        "e2e": {"value": round(shape.T * world / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": shape.T * shape.H * 2 + (0 if args.gated else shape.T * shape.E * 4),
                "d2h_bytes_per_step": shape.T * shape.H * 2},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "shared_overlap": overlap,
    }
    if (args.workload == "decode" and not (args.no_prefill or args.experts or args.dtype or args.gated
                                            or args.shared_fold or args.eager) and world == 1):
        result["prefill"] = measure_prefill(moe, synth, w, dev, main, peaks)
    if gemm_ab is not None:
        result["gemm_mode_ab"] = gemm_ab
    if option_ab is not None:
        result["option_ab"] = option_ab
    if rank == 0 and not args.no_cpu_baseline:
        import oracle

        rate, n, dt, thr = cpu_oracle_rate(shape, x, logits, w, budget_s=12.0)
        result["cpu_baseline"] = {"value": round(rate, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                  "sample": f"{n} tokens of the {args.workload} workload (its {shape.T} tokens "
                                            f"cycled) through the fp64 oracle ({dt:.1f} s)"}
        # The same oracle on one thread: this workload (bounded sample) and
        # the whole tiny layer.
        oracle.set_num_threads(1)
        try:
            single = {}
            r1, n1, dt1, _ = cpu_oracle_rate(shape, x, logits, w, budget_s=6.0)
            single[args.workload] = {"value": round(r1, 3), "unit": "tokens/s",
                                     "sample": f"{n1} tokens ({dt1:.1f} s)"}
            tiny = synth.WORKLOADS["tiny"]
            xt, lt = synth.make_activations(tiny, seed=0)
            wt = synth.make_weights(tiny, seed=0)
            rt, nt, dtt, _ = cpu_oracle_rate(tiny, xt, lt, wt, budget_s=0.5, max_tokens=tiny.T)
            single["tiny"] = {"value": round(rt, 3), "unit": "tokens/s",
                              "sample": f"the whole tiny layer ({nt} tokens, {dtt * 1e3:.2f} ms)"}
            result["cpu_baseline"]["single_thread"] = single
        finally:
            oracle.set_num_threads(thr)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_reference(args):
    import numpy as np
    import torch

    import oracle
    import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shape = synth.WORKLOADS[args.workload]
    if args.dtype:
        shape = shape.with_(dtype=args.dtype)
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    x, logits = synth.make_activations(shape, device=dev, seed=0)
    w = synth.make_weights(shape, device=dev, seed=0)
    run = oracle_layer_fn(shape, x, logits, w)
    del w

    def step(n):
        run((np.arange(n) % shape.T).astype(np.int32))

    t0 = time.perf_counter()
    step(1)
    t1 = time.perf_counter() - t0
    total_budget = 150.0  # seconds for warmup + timed steps
    n = max(1, min(shape.T, int(total_budget / max(1, args.steps + args.warmup) / max(t1, 1e-6))))
    for _ in range(args.warmup):
        step(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(n)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = n / (ms * 1e-3)
    thr = oracle.num_threads()
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64" + (f" on {shape.dtype} operands" if shape.dtype != "bf16" else ""),
        "data": "synthetic (same seeds as the CUDA arm)",
        "config": {"workload": f"Hy3-shape {args.workload} MoE layer" + (f", {args.dtype} operands" if args.dtype else ""),
                   "T": shape.T, "H": shape.H, "E": shape.E,
                   "K": shape.K, "I": shape.I, "I_shared": shape.I_shared},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                         "sample": f"{n} token(s) of the {args.workload} workload per step through the fp64 oracle"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
