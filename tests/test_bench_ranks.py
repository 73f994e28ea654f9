"""The bench's multi-rank aggregation on CPU: two gloo ranks, replicas-only scaling.

Each rank reports its own step time; the job's time is the slowest rank's (max over
ranks), and the whole-job throughput is world_size x per-rank work / that time.  The
GPU path runs the same function over NCCL.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
        ms, value = bench.replica_throughput(local_ms, 3.0, world, dist, "cpu")
        results[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        got = dict(results)
    assert codes == [0, 0], codes
    for r in range(world):
        ms, value = got[r]
        assert ms == pytest.approx(20.0)
        assert value == pytest.approx(3.0 * 2 / 0.020)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.replica_throughput(4.0, 2.0, 1)
    assert ms == 4.0 and value == pytest.approx(500.0)
