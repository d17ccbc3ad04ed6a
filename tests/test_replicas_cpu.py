"""The multi-GPU path is replicas only (no exchange step on the KDA path):
N ranks run independent copies and rank 0 reports every rank's tokens over
the slowest rank's time.  These checks run the cross-rank reduction of
bench.py on CPU with two gloo ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms for phase 0 and 5 ms for phase 1
        got = bench.max_over_ranks([rank + 1.0, 5.0], world)
        value = bench.replica_throughput(4096, 10, world, got[0] / 1e3)
        q.put((rank, got, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in out:
        assert got == [2.0, 5.0]  # the slowest rank's times, on every rank
        assert value == pytest.approx(4096 * 10 * 2 / 2e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.replica_throughput(4096, 10, 1, 0.5) == pytest.approx(81920.0)
