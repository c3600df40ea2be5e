"""The N>1 path of bench.py (independent replicas, barrier + max-over-ranks
timing) on CPU with the gloo backend, world size 2."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [1.5, 2.5][rank]
    ms = bench.reduce_max(local_ms, world)
    val = bench.job_value(1e12, world, ms)
    dist.barrier()
    q.put((rank, ms, val))
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, val in res:
        assert ms == 2.5                      # the slowest rank's time, on every rank
        assert val == pytest.approx(2 * 1e12 / 2.5e-3 / 1e12)  # both ranks' work / that time


def test_single_rank_helpers():
    import bench
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.job_value(2e12, 1, 2.0) == pytest.approx(1000.0)
