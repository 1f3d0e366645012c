"""The multi-rank path of bench.py (replicas, no data-path collective): the
slowest rank's time and the whole-job token count, over gloo with two ranks
on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms_local = [1.5, 2.0][rank]
    value, ms = bench.aggregate(64, ms_local, world, torch.device("cpu"))
    bench.barrier(world)
    q.put((rank, value, ms))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, value, ms in res:
        assert ms == 2.0
        assert value == pytest.approx(64 * 2 / 2e-3)


def test_single_rank_needs_no_process_group():
    import bench

    value, ms = bench.aggregate(64, 1.25, 1, torch.device("cpu"))
    assert ms == 1.25 and value == pytest.approx(64 / 1.25e-3)


def _run_bench(args, env_extra=None):
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], cwd=root, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    return [json.loads(l) for l in lines]


def test_reference_arm_prints_one_contract_line():
    # The reference arm is the oracle on the host cores: it runs without a GPU.
    (line,) = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    assert _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                      {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
