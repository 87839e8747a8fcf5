"""The multi-process path of the benchmark on CPU: two gloo ranks, each an
independent replica, agree on the slowest rank's time, and the whole-job
throughput counts every rank's work.  (The path shards by request with no
exchange step, so no collective touches the data.)"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(1.5 + rank, world, "cpu")      # rank 1 is the slow one
        results[rank] = (t, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == 2.5
    assert results[0][1] == (2, 0, 0) and results[1][1] == (2, 1, 1)


def test_single_rank_is_identity_and_throughput_counts_every_rank():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    one = bench.job_throughput_gbs(10**9, 10, 1, 2.0)
    assert one == pytest.approx(5.0)
    assert bench.job_throughput_gbs(10**9, 10, 4, 2.0) == pytest.approx(4 * one)   # weak scaling
