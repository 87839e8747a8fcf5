"""The two decode consumers against the fp64 oracle.

libshkv has two consumers for the same decode step: warp-level mma.sync
tiles and, for head dim 128, tcgen05 tiles with tokens along the MMA's M
dimension and the accumulators in tensor memory.  A pool names one with
shkv_pool_set_decode_consumer; these tests force the tcgen05 consumer on every row
count class (padded N of 16, 32, 48 and 64; three- and two-stage rings;
4 and 8 pages per 128-token stage), check that it is the one that ran, and
compare with the oracle and with the invariants the definition fixes.  The
automatic choice takes tcgen05 from 16 stacked rows up; the last tests
force mma.sync there so both consumers stay covered at every row count.
"""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import CONSUMER, bits_to_torch, compare, make_pool, oracle_for_requests, torch_to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture
def umma():
    CONSUMER["name"] = "umma"
    yield
    CONSUMER["name"] = "auto"


SHAPES = {
    "qwen14b": dict(N=8, Hq=40, Hkv=8, D=128, P=32),     # R = 40: N 48, 3 stages, 4 pages per stage
    "r40_p16": dict(N=8, Hq=40, Hkv=8, D=128, P=16),     # R = 40, 8 pages per stage
    "long": dict(N=8, Hq=16, Hkv=8, D=128, P=16),        # R = 16
    "llama8b": dict(N=2, Hq=32, Hkv=8, D=128, P=16),     # R = 8
    "r24": dict(N=3, Hq=64, Hkv=8, D=128, P=32),         # R = 24: N 32
    "r64": dict(N=8, Hq=16, Hkv=2, D=128, P=16),         # R = 64: N 64, 2 stages
    "r1": dict(N=1, Hq=8, Hkv=8, D=128, P=32),           # R = 1
}


def run(wl, q, k, v, what):
    pool = make_pool(wl, k, v)
    assert pool.decode_consumer(wl.N, wl.Hq) == "tcgen05"
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what=what)
    return pool, out, lse


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_umma_consumer_matches_oracle(umma, shape):
    lens = [1, 15, 16, 17, 33, 127, 128, 129, 257, 1000, 2049, 4100]
    wl = W.custom_workload(shape, B=len(lens), lens_prefill=lens, seed=23, **SHAPES[shape])
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    run(wl, q, k, v, f"umma {shape}")


def test_head_dim_64_stays_on_mma_sync(umma):
    wl = W.custom_workload("d64", B=3, N=3, Hq=64, Hkv=8, D=64, P=32, lens_prefill=[5, 300, 2000], seed=3)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    assert pool.decode_consumer(wl.N, wl.Hq) == "mma.sync"
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what="d64")


@pytest.mark.parametrize("P", [16, 32])
def test_umma_long_single_request_split_and_merged(umma, P):
    wl = W.custom_workload("split", B=1, N=8, Hq=40, Hkv=8, D=128, P=P, lens_prefill=[60000], seed=4)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    run(wl, q, k, v, f"umma split P={P}")


def test_umma_large_scores_exercise_the_lazy_rescale(umma):
    """Keys grow along the sequence so a row's running max rises by far more
    than 2^10 (base 2) between early and late stages: O and the row sums in
    tensor memory must be rescaled on the fly.  (Far more peaked inputs
    would hit the bf16 rounding bound of P, about 2^-8 * max|V|, rather than
    the 1e-2 bar.)"""
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
    run(wl, q, k, v, "umma rescale")


def test_umma_identical_queries_give_identical_slices(umma):
    wl = W.custom_workload("ident", B=3, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[700, 3000, 64], seed=2)
    q = W.gen_q(wl)
    for m in range(1, wl.N):
        q[:, m * wl.Hq:(m + 1) * wl.Hq] = q[:, :wl.Hq]
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, return_lse=True)
    for m in range(1, wl.N):
        assert torch.equal(out[:, m * wl.Hq:(m + 1) * wl.Hq], out[:, :wl.Hq])
        assert torch.equal(lse[:, m * wl.Hq:(m + 1) * wl.Hq], lse[:, :wl.Hq])


def test_umma_page_permutation_gives_identical_bits(umma):
    wl = W.custom_workload("perm", B=4, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[700, 3000, 64, 9000], seed=6)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    out1 = make_pool(wl, k, v).decode_attention(bits_to_torch(q), wl.N)
    perm = np.random.default_rng(5).permutation(wl.num_pages)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    wl2 = W.Workload(**{**wl.__dict__})
    wl2.block_table = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    out2 = make_pool(wl2, k2, v2).decode_attention(bits_to_torch(q), wl.N)
    assert torch.equal(out1, out2)


def test_umma_single_key_returns_v_exactly(umma):
    wl = W.custom_workload("one", B=3, N=8, Hq=40, Hkv=8, D=128, P=16, lens_prefill=[1, 1, 1], seed=8)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    got = torch_to_bits(pool.decode_attention(bits_to_torch(q), wl.N))
    for b in range(wl.B):
        page = wl.block_table[b, 0]
        for r in range(wl.rows):
            np.testing.assert_array_equal(got[b, r], v[page, (r % wl.Hq) // wl.G, 0])


def test_umma_equal_scores_return_mean_of_values(umma):
    lens = [5, 16, 100, 1234]
    wl = W.custom_workload("mean", B=len(lens), N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=lens, seed=12)
    q = W.gen_q(wl)
    q[:] = 0
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, return_lse=True)
    vf = W.f32_from_bf16_bits(v).astype(np.float64)
    for b, L in enumerate(lens):
        t = np.arange(L)
        vb = vf[wl.block_table[b, t // wl.P], :, t % wl.P, :]
        ref = np.stack([vb[:, (r % wl.Hq) // wl.G].mean(0) for r in range(wl.rows)])
        compare(out[b], ref, what=f"mean b={b}")
        np.testing.assert_allclose(lse[b].cpu().numpy(), np.log(L), atol=1e-4)


def test_umma_shared_equals_unshared_per_model_runs(umma):
    wl = W.custom_workload("unsh", B=4, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[700, 3000, 64, 9000], seed=13)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    qt = bits_to_torch(q)
    shared = pool.decode_attention(qt, wl.N)
    for m in range(wl.N):
        single = pool.decode_attention(qt[:, m * wl.Hq:(m + 1) * wl.Hq].contiguous(), 1)
        compare(shared[:, m * wl.Hq:(m + 1) * wl.Hq], single.double().cpu().numpy(), what=f"m={m}")


def test_umma_out_of_range_page_sets_flag_and_is_skipped(umma):
    wl = W.custom_workload("oob", B=2, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[300, 300], seed=14)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    ref = pool.decode_attention(bits_to_torch(q), wl.N).clone()
    assert pool.check_errors() == 0
    pool.block_table[1, 3] = wl.num_pages + 7
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    assert pool.check_errors() & N.SHKV_ERRF_PAGE_OOB
    assert torch.equal(out[0], ref[0])
    assert bool(torch.isfinite(out.float()).all())


def test_umma_device_length_disagreeing_with_host_copy_sets_flag(umma):
    wl = W.custom_workload("len", B=2, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[300, 300], seed=15)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    pool.seq_lens[0] = 17
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    assert pool.check_errors() & N.SHKV_ERRF_SEQ_LEN
    assert bool(torch.isfinite(out.float()).all())


def test_umma_full_size_qwen14b_sampled(umma):
    wl = W.make_workload("qwen14b")
    q = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl)
    pool = make_pool(wl, k_dev, v_dev)
    assert pool.decode_consumer(wl.N, wl.Hq) == "tcgen05"
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    order = np.argsort(wl.lens_final)
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    for b, (ref, lref) in oracle_for_requests(wl, q, k_dev, v_dev, picks).items():
        compare(out[b], ref, lse[b], lref, what=f"umma qwen14b b={b}")


# --------------------------------------------------------------------------
# the mma.sync consumer where the automatic choice is tcgen05
# --------------------------------------------------------------------------
@pytest.fixture
def mma():
    CONSUMER["name"] = "mma"
    yield
    CONSUMER["name"] = "auto"


def test_automatic_choice_by_rows_and_head_dim():
    for shape, want in [("qwen14b", "tcgen05"), ("r24", "tcgen05"), ("r64", "tcgen05"), ("long", "tcgen05"),
                        ("llama8b", "mma.sync"), ("r1", "mma.sync")]:
        sh = SHAPES[shape]
        wl = W.custom_workload(shape, B=1, lens_prefill=[40], seed=1, **sh)
        k, v = W.gen_pool(wl)
        assert make_pool(wl, k, v).decode_consumer(wl.N, wl.Hq) == want, shape


@pytest.mark.parametrize("shape", ["qwen14b", "r40_p16", "r64", "long", "r24"])
def test_mma_consumer_matches_oracle_for_many_rows(mma, shape):
    lens = [1, 17, 129, 1000, 4100]
    wl = W.custom_workload(shape, B=len(lens), lens_prefill=lens, seed=29, **SHAPES[shape])
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    assert pool.decode_consumer(wl.N, wl.Hq) == "mma.sync"
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what=f"mma {shape}")


def test_mma_long_single_request_split_and_merged(mma):
    wl = W.custom_workload("split", B=1, N=8, Hq=40, Hkv=8, D=128, P=32, lens_prefill=[60000], seed=4)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    assert pool.decode_consumer(wl.N, wl.Hq) == "mma.sync"
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    compare(out, ref, lse, lref, what="mma split")


def test_consumer_setting_is_per_pool_and_checked():
    """A pool's consumer choice applies to that pool only; unknown values are
    rejected by the binding and by the C entry point."""
    sh = SHAPES["long"]
    wl = W.custom_workload("setting", B=1, lens_prefill=[40], seed=1, **sh)
    k, v = W.gen_pool(wl)
    a, b = make_pool(wl, k, v), make_pool(wl, k, v)
    a.set_decode_consumer("mma")
    assert a.decode_consumer(wl.N, wl.Hq) == "mma.sync"
    assert b.decode_consumer(wl.N, wl.Hq) == "tcgen05"
    a.set_decode_consumer("auto")
    assert a.decode_consumer(wl.N, wl.Hq) == "tcgen05"
    with pytest.raises(ValueError):
        a.set_decode_consumer("fastest")
    with pytest.raises(N.ShkvError) as e:
        N.shkv_pool_set_decode_consumer(a.handle, 7)
    assert e.value.status == N.SHKV_ERR_INVALID_ARG
