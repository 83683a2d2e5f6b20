"""The benchmark's multi-replica host logic on CPU: two gloo ranks (one
process each, as torchrun starts them) agree on the slowest rank's time and
on the whole-job throughput; a rank that raises is reported, not hung on."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results, fail_rank):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=__import__("datetime").timedelta(seconds=20))
    try:
        if rank == fail_rank:
            raise RuntimeError("replica failed before its first step")
        ms = bench.max_over_ranks(torch, dist, 1.0 + rank, torch.device("cpu"))
        results[rank] = (ms, bench.job_gbs(1e9, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world, fail_rank=-1):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, results, fail_rank))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    return dict(results), codes


def test_two_replicas_take_the_slowest_time():
    results, codes = _run(2)
    assert codes == [0, 0]
    assert results[0][0] == results[1][0] == 2.0        # max of 1.0 and 2.0 ms
    assert results[0][1] == pytest.approx(2 * 1e9 / 2e-3 / 1e9)  # 1000 GB/s


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, None, 3.5, None) == 3.5
    assert bench.job_gbs(2e9, 1, 1.0) == pytest.approx(2000.0)


def test_a_failing_replica_ends_the_job():
    _, codes = _run(2, fail_rank=1)
    assert codes[1] != 0          # the failing rank exits with an error
    assert all(c is not None for c in codes), "a rank hung"
