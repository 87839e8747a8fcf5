"""Request sharding across replicas (PrefillShare framework scope: decode runs
in a data-parallel pool of GPUs), on the CPU.

shkv_partition_requests divides a batch among world_size replicas by unique
KV pages, longest request first, each to the replica holding the fewest
pages.  Checked here: every request goes to exactly one replica, the
per-replica page counts add up, the heaviest replica is within the greedy
bound (mean + largest request), the assignment is deterministic, and -- with
two gloo ranks, each running the oracle on its own shard only -- the shards'
results put back in request order equal the unsharded oracle bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import build as B
from cross_model_shared_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return N.load()


def _pages(lens, P):
    return (np.asarray(lens, np.int64) + P - 1) // P


@pytest.mark.parametrize("seed,batch,ws,P", [(0, 128, 2, 32), (1, 128, 8, 32), (2, 37, 3, 16), (3, 5, 8, 16),
                                             (4, 1024, 4, 16), (5, 1, 1, 16)])
def test_partition_covers_every_request_once_within_the_greedy_bound(seed, batch, ws, P):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 70000, size=batch).astype(np.int32)
    owner, rank_pages = N.shkv_partition_requests(lens, P, ws)
    pages = _pages(lens, P)
    assert owner.shape == (batch,) and ((owner >= 0) & (owner < ws)).all()
    for r in range(ws):
        assert rank_pages[r] == pages[owner == r].sum()
    assert rank_pages.sum() == pages.sum()
    assert rank_pages.max() <= pages.sum() / ws + pages.max()
    if batch >= ws:
        assert (np.bincount(owner, minlength=ws) > 0).all()
    again, _ = N.shkv_partition_requests(lens, P, ws)
    assert np.array_equal(owner, again)


def test_partition_examples_by_hand():
    # pages 7, 1, 4, 4, 2 (P = 16), longest first: 7 -> r0; 4 -> r1; 4 -> r1 (4 < 7); 2 -> r0 (7 < 8); 1 -> r1 (8 < 9)
    lens = np.array([112, 3, 64, 50, 20], np.int32)
    owner, rank_pages = N.shkv_partition_requests(lens, 16, 2)
    assert owner.tolist() == [0, 1, 1, 1, 0]
    assert rank_pages.tolist() == [9, 9]
    owner, rank_pages = N.shkv_partition_requests(lens, 16, 1)
    assert owner.tolist() == [0] * 5 and rank_pages.tolist() == [18]
    owner, rank_pages = N.shkv_partition_requests(lens[:2], 16, 4)     # more replicas than requests
    assert owner.tolist() == [0, 1] and rank_pages.tolist() == [7, 1, 0, 0]


def test_partition_rejects_bad_arguments(lib):
    lens = np.array([5, -1], np.int32)
    with pytest.raises(N.ShkvError):
        N.shkv_partition_requests(lens, 16, 2)
    with pytest.raises(N.ShkvError):
        N.shkv_partition_requests(np.array([5], np.int32), 16, 0)
    with pytest.raises(N.ShkvError):
        N.shkv_partition_requests(np.array([5], np.int32), 0, 2)


def test_replica_batches_are_new_draws_of_the_same_mix():
    a, b = W.make_workload("qwen14b"), W.make_workload("qwen14b", 1)
    assert np.array_equal(a.lens_final, W.make_workload("qwen14b", 0).lens_final)
    assert not np.array_equal(a.lens_final, b.lens_final)
    assert a.B == b.B and b.lens_final.min() >= 1024 and b.lens_final.max() <= 65536


# --------------------------------------------------------------------------
# two gloo ranks, each with its own shard
# --------------------------------------------------------------------------
SHAPE = dict(N=2, Hq=8, Hkv=2, D=64, P=16)


def _global_problem():
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 600, size=13).astype(np.int32)
    wl = W.custom_workload("shards", B=len(lens), lens_prefill=lens, seed=9, **SHAPE)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    return wl, q, k, v


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        N.load()
        wl, q, k, v = _global_problem()
        owner, rank_pages = N.shkv_partition_requests(wl.lens_final, wl.P, world)
        owners = [None] * world
        dist.all_gather_object(owners, owner.tolist())
        mine = np.flatnonzero(owner == rank)
        # this rank holds only its own requests' pages, renumbered 0..n-1
        bt_rows, pages = [], []
        for b in mine:
            npg = int(_pages([wl.lens_final[b]], wl.P)[0])
            bt_rows.append(np.arange(len(pages), len(pages) + npg, dtype=np.int32))
            pages.extend(int(x) for x in wl.block_table[b, :npg])
        width = max(1, max((len(r) for r in bt_rows), default=1))
        bt = np.full((len(mine), width), -1, np.int32)
        for i, r in enumerate(bt_rows):
            bt[i, :len(r)] = r
        ids = np.asarray(pages, dtype=np.int64)
        out, lse = oracle.decode_attention(q[mine], k[ids], v[ids], bt, wl.lens_final[mine], n_models=wl.N,
                                           hq=wl.Hq, scale=wl.scale)
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine.tolist(), out, lse, int(ids.size)))
        results[rank] = (owners, gathered, rank_pages.tolist())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shards_reassemble_to_the_unsharded_oracle():
    import oracle
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    owners, gathered, rank_pages = results[0]
    assert owners[0] == owners[1], "ranks computed different assignments"
    wl, q, k, v = _global_problem()
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    seen = []
    out = np.zeros_like(ref)
    lse = np.zeros_like(lref)
    for r, (mine, o, l, npages) in enumerate(gathered):
        assert npages == rank_pages[r]
        seen += mine
        out[mine], lse[mine] = o, l
    assert sorted(seen) == list(range(wl.B)), "every request exactly once"
    pages = _pages(wl.lens_final, wl.P)
    assert max(rank_pages) <= pages.sum() / 2 + pages.max()
    assert np.array_equal(out, ref) and np.array_equal(lse, lref)
