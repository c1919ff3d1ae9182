"""The N > 1 path of bench.py on CPU: two gloo ranks, each an independent replica.

The hot path has no exchange step, so a multi-GPU run is N replicas of the
one-GPU step.  What the ranks share is host-side bookkeeping: every per-step
time is maximised over the ranks (the job is as slow as its slowest replica)
and the job's rate is all ranks' units over that time.  These tests run that
bookkeeping as two gloo processes on 127.0.0.1.
"""

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


def _rank_main(rank, world, port, times_by_rank, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(times_by_rank[rank], world, "cpu")
        dist.barrier()
        results[rank] = got
    finally:
        dist.destroy_process_group()


def _run(times_by_rank):
    world = len(times_by_rank)
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, times_by_rank, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0] * world, codes
        return [list(results[r]) for r in range(world)]


def test_max_over_two_gloo_ranks():
    times = [[1.5e-4, 1.1e-4, 4.0e-5, 5.0e-5, 9.0e-4], [1.7e-4, 1.0e-4, 6.0e-5, 5.0e-5, 8.0e-4]]
    got = _run(times)
    want = [max(a, b) for a, b in zip(*times)]
    assert got[0] == want and got[1] == want


def test_single_rank_is_unchanged():
    t = [1.0, 2.5, 3]
    assert bench.max_over_ranks(t, 1, "cpu") == [1.0, 2.5, 3.0]


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_job_throughput_counts_every_replica(world):
    # 32768 KV tokens per replica, slowest replica 0.2 ms
    assert bench.job_throughput(32768, world, 2e-4) == pytest.approx(32768 * world / 2e-4)
