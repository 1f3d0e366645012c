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
