"""The tcgen05 (tensor-memory) consumer against the fp64 oracle.

libshkv has two consumers for the same decode step: warp-level mma.sync
tiles (the default) and tcgen05 tiles with accumulators in tensor memory.
SHKV_DECODE_CONSUMER selects one per call; these tests force the tcgen05
consumer on every supported shape class and compare with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, make_pool, oracle_for_requests

pytestmark = pytest.mark.gpu


@pytest.fixture
def umma(monkeypatch):
    monkeypatch.setenv("SHKV_DECODE_CONSUMER", "umma")


SHAPES = {
    "qwen14b": dict(N=8, Hq=40, Hkv=8, D=128, P=32),     # R = 40
    "long": dict(N=8, Hq=16, Hkv=8, D=128, P=16),        # R = 16
    "llama8b": dict(N=2, Hq=32, Hkv=8, D=128, P=16),     # R = 8
    "r64": dict(N=8, Hq=16, Hkv=2, D=128, P=16),         # R = 64
    "r24_d64": dict(N=3, Hq=64, Hkv=8, D=64, P=32),      # R = 24, head dim 64
    "r1": dict(N=1, Hq=8, Hkv=8, D=128, P=32),           # R = 1
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_umma_consumer_matches_oracle(umma, shape):
    lens = [1, 15, 16, 17, 33, 257, 1000, 2049, 4100]
    wl = W.custom_workload(shape, B=len(lens), lens_prefill=lens, seed=23, **SHAPES[shape])
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what=f"umma {shape}")


def test_umma_long_single_request_split_and_merged(umma):
    wl = W.custom_workload("split", B=1, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[60000], seed=4)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what="umma split")


def test_umma_large_scores_exercise_the_lazy_rescale(umma):
    """Keys grow along the sequence so a row's running max rises by more
    than 2^8 (base 2) between early and late tiles: the tensor-memory O must
    be rescaled on the fly.  (Far more peaked inputs would hit the bf16
    rounding bound of P, about 2^-8 * max|V|, rather than the 1e-2 bar.)"""
    lens = [3000, 777]
    wl = W.custom_workload("rescale", B=2, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=lens, seed=9)
    q = W.bf16_bits_from_f32(2.0 * W.f32_from_bf16_bits(W.gen_q(wl)))
    k, v = W.gen_pool(wl)
    kf = W.f32_from_bf16_bits(k)
    for b, L in enumerate(lens):
        for t in range(L):
            page, slot = wl.block_table[b, t // wl.P], t % wl.P
            kf[page, :, slot] *= 0.25 + 1.5 * t / L
    k = W.bf16_bits_from_f32(kf)
    pool = make_pool(wl, k, v)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what="umma rescale")


def test_umma_identical_queries_give_identical_slices(umma):
    wl = W.custom_workload("ident", B=3, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[700, 3000, 64], seed=2)
    q = W.gen_q(wl)
    for m in range(1, wl.N):
        q[:, m * wl.Hq:(m + 1) * wl.Hq] = q[:, :wl.Hq]
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    for m in range(1, wl.N):
        assert torch.equal(out[:, m * wl.Hq:(m + 1) * wl.Hq], out[:, :wl.Hq])


def test_umma_full_size_qwen14b_sampled(umma):
    wl = W.make_workload("qwen14b")
    q = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl)
    pool = make_pool(wl, k_dev, v_dev)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    order = np.argsort(wl.lens_final)
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    for b, (ref, lref) in oracle_for_requests(wl, q, k_dev, v_dev, picks).items():
        compare(out[b], ref, lse[b], lref, what=f"umma qwen14b b={b}")
