"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The aggregation shards over tokens with no exchange: N GPUs run N independent
replicas (weak scaling). What N > 1 adds is host-side: joining the process
group, the barrier around the timed region, and taking the slowest rank's step
time. These run here as two gloo ranks on 127.0.0.1.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r, w, local = bench.dist_setup(world, backend="gloo")
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(times[rank], w)
    value = bench.job_throughput(8192, w, slowest)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((rank, slowest, value))


def test_two_gloo_ranks_take_the_slowest_step():
    world, port = 2, _free_port()
    times = [5.0, 7.5]  # ms per step seen by rank 0 and rank 1
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == 7.5
        assert value == pytest.approx(8192 * 2 / 7.5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.dist_setup(1) == (0, 1, 0)
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(100, 1, 1.0) == pytest.approx(1e5)
