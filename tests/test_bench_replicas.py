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


def test_tensor_roofline_blends_mxfp8_and_bf16_peaks():
    """BF16: every FLOP at the BF16 peak.  MXFP8: routed FLOPs at twice the
    BF16 peak, the BF16 shared expert's at once, so the time at peak is
    routed / 2P + shared / P (DSV3: 1.1545e13 + 1.443e12 FLOP)."""
    import bench
    import moe_inputs as mi
    P = 1000.0
    bf = bench.tensor_roofline(mi.CONFIGS["dsv3"], 20.0, P, "test", P)
    assert bf["peak"] == pytest.approx(P)
    assert bf["frac"] == pytest.approx(mi.CONFIGS["dsv3"].flops() / 0.020 / 1e12 / P)
    mx = bench.tensor_roofline(mi.CONFIGS["dsv3_mxfp8"], 10.0, P, "test", 2 * P)
    routed, shared = 6.0 * 16384 * 8 * 7168 * 2048, 6.0 * 16384 * 7168 * 2048
    t_peak = routed / (2 * P * 1e12) + shared / (P * 1e12)
    assert mx["frac"] == pytest.approx(t_peak / 0.010)
    assert mx["frac_of_burst_peak"] == pytest.approx(mx["frac"] / 2)
    assert P < mx["peak"] < 2 * P


def test_phase_bandwidths_from_stamps():
    import bench
    import moe_inputs as mi
    s = mi.CONFIGS["dsv3"]
    res = {"router_ms": [0.1, 0.1], "phase_stamps_ms": {"last_fill": 5.0, "combine_start": 10.0,
                                                         "combine_end": 10.5}}
    bw = bench.phase_bandwidths(s, res, 6000.0)
    comb = (s.T * 9 * s.D * 2 + s.T * s.D * 2 + s.T * s.k * 4)
    assert bw["combine"]["GB/s"] == pytest.approx(comb / 0.5e-3 / 1e9)
    assert bw["ring_fill"]["GB/s"] == pytest.approx(s.T * s.k * s.D * 4 / 5e-3 / 1e9)
    assert bw["router"]["GB/s"] == pytest.approx((s.T * s.D * 2 + s.E * s.D * 2) / 0.1e-3 / 1e9)
    none = bench.phase_bandwidths(s, {"router_ms": [0.1], "phase_stamps_ms": {"last_fill": None,
                                                                               "combine_start": None,
                                                                               "combine_end": None}}, 6000.0)
    assert "combine" not in none and "ring_fill" not in none
