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


def test_reference_arm_prints_one_contract_line():
    """The reference arm (the fp64 oracle on the host cores) needs no GPU: one
    JSON line with the main line's metric and unit, `impl: reference`, and the
    cpu_baseline and e2e objects that describe it."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["value"] > 0 and d["config"]["workload"] == "tiny"
    import argparse
    gpu_arm_config = bench.workload_config(bench.Job(argparse.Namespace(config="tiny", batch=0), 1, 0,
                                                     partition=False))
    assert d["config"] == gpu_arm_config             # the same keys and values as the GPU arm's line
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_prints_once():
    """Launched like the multi-GPU bench (torchrun, two ranks), the reference
    arm runs on rank 0 alone: one JSON line, and every rank exits 0."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--config", "tiny", "--gpus", "2",
           "--steps", "2", "--warmup", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    assert len([l for l in out.stdout.splitlines() if l.startswith("{")]) == 1


def test_job_shards_the_global_batch_by_the_partitioner():
    """Under torchrun the bench's global batch is N batches of the workload;
    each rank's local workload holds exactly its requests (by the library's
    partitioner), and the ranks' step bytes add up to the job's."""
    import argparse

    import numpy as np

    from cross_model_shared_gb300 import build as B
    B.build()
    args = argparse.Namespace(config="qwen14b", batch=0)
    one = bench.Job(args, 1, 0)
    assert one.local is one.base and one.total_bytes() == bench.step_bytes(one.base)
    jobs = [bench.Job(args, 4, r) for r in range(4)]
    j0 = jobs[0]
    assert len(j0.lens_final) == 4 * j0.base.B
    assert np.array_equal(j0.lens_final[:j0.base.B], one.lens_final)
    got = sorted(np.concatenate([j.local.lens_final for j in jobs]).tolist())
    assert got == sorted(j0.lens_final.tolist())
    for r, j in enumerate(jobs):
        assert np.array_equal(j.owner, j0.owner)
        assert bench.step_bytes(j.local) == j0.rank_bytes()[r]
    assert sum(j0.rank_bytes()) == j0.total_bytes()
    cfg = bench.workload_config(j0)
    assert cfg["batch"] == 4 * j0.base.B and cfg["workload"] == "qwen14b"
    assert cfg == bench.workload_config(bench.Job(args, 4, 0, partition=False))
