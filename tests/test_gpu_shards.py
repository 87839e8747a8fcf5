"""Request shards (PrefillShare framework scope: decode on a data-parallel
pool of GPUs) through the CUDA path, on one GPU.

shkv_partition_requests divides a batch among replicas; each replica holds
only its own requests' pages (renumbered into a pool of its own, with its
own block table) and decodes them.  Here every shard runs on the one GPU in
turn: each shard's outputs match the oracle, every request is decoded by
exactly one shard, and the shards put back in request order match the
unsharded decode within the parity bar (the split plans differ, so the
summation order may too).
"""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, make_pool

pytestmark = pytest.mark.gpu


def _shard(wl, q, k, v, mine, seed):
    """The workload of requests `mine`, its pages copied out of the global
    pool into a pool of their own in a fresh random order."""
    lens = wl.lens_final[mine]
    sub = W.custom_workload("shard", B=len(mine), N=wl.N, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D, P=wl.P,
                            lens_prefill=lens, seed=seed)
    ks = np.empty((sub.num_pages,) + k.shape[1:], k.dtype)
    vs = np.empty_like(ks)
    for i, b in enumerate(mine):
        npg = int((wl.lens_final[b] + wl.P - 1) // wl.P)
        ks[sub.block_table[i, :npg]] = k[wl.block_table[b, :npg]]
        vs[sub.block_table[i, :npg]] = v[wl.block_table[b, :npg]]
    return sub, np.ascontiguousarray(q[mine]), ks, vs


@pytest.mark.parametrize("shape,ws", [
    (dict(N=4, Hq=32, Hkv=8, D=128, P=16), 3),      # Qwen3-8B heads, tcgen05 consumer
    (dict(N=2, Hq=32, Hkv=8, D=128, P=16), 4),      # Llama-3.1-8B heads, mma.sync consumer
])
def test_shards_match_unsharded_decode_and_oracle(shape, ws):
    rng = np.random.default_rng(61)
    lens = rng.integers(1, 6000, size=26).tolist()
    wl = W.custom_workload("global", B=len(lens), lens_prefill=lens, seed=62, **shape)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    full, full_lse = make_pool(wl, k, v).decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    owner, rank_pages = N.shkv_partition_requests(wl.lens_final, wl.P, ws)
    pages = (wl.lens_final.astype(np.int64) + wl.P - 1) // wl.P
    assert rank_pages.max() <= pages.sum() / ws + pages.max()
    seen = []
    for r in range(ws):
        mine = np.flatnonzero(owner == r)
        assert len(mine) > 0
        seen += mine.tolist()
        sub, qs, ks, vs = _shard(wl, q, k, v, mine, seed=70 + r)
        assert int(((sub.lens_final.astype(np.int64) + wl.P - 1) // wl.P).sum()) == rank_pages[r]
        pool = make_pool(sub, ks, vs)
        out, lse = pool.decode_attention(bits_to_torch(qs), sub.N, scale=sub.scale, return_lse=True)
        assert pool.check_errors() == 0
        ref, lref = oracle.decode_attention(qs, ks, vs, sub.block_table, sub.lens_final, n_models=sub.N,
                                            hq=sub.Hq, scale=sub.scale)
        compare(out, ref, lse, lref, what=f"shard {r}")
        idx = torch.as_tensor(mine, device=full.device)
        compare(out, full.index_select(0, idx).double().cpu().numpy(), lse,
                full_lse.index_select(0, idx).double().cpu().numpy(), what=f"shard {r} vs unsharded")
    assert sorted(seen) == list(range(wl.B))
