"""The multi-process side of bench.py on CPU (gloo, world size 2): the layer
has no data-parallel exchange on one node, so N GPUs run N independent
replicas; the timed region's length is the slowest rank's, and the whole-job
throughput counts every replica's tokens."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.reduce_max(10.0 + 5.0 * rank, world)
    value = bench.replica_throughput(world, 16384, 4, slowest)
    dist.barrier()
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 16384 * 4 / 0.015)


def test_single_process_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.replica_throughput(1, 100, 10, 1000.0) == pytest.approx(1000.0)
