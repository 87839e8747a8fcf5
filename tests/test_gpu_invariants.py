"""GPU invariants the definition fixes, checked on the CUDA path itself, and
the library's error reporting (host argument checks and device error bits
raised by the kernels' own bounds checks)."""
import numpy as np
import pytest
import torch

from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, make_pool, torch_to_bits

pytestmark = pytest.mark.gpu


def setup(lens, seed=21, **shape):
    wl = W.custom_workload("inv", B=len(lens), lens_prefill=lens, seed=seed, **shape)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    return wl, q, k, v, make_pool(wl, k, v)


LLAMA = dict(N=2, Hq=32, Hkv=8, D=128, P=16)
QWEN14 = dict(N=8, Hq=40, Hkv=8, D=128, P=32)


@pytest.mark.parametrize("shape", [LLAMA, QWEN14])
def test_identical_query_sets_give_identical_slices(shape):
    """ICaRus key design 2: one identical cache, so decoders with equal
    queries get bit-identical outputs."""
    wl, q, k, v, pool = setup([700, 3000, 64, 9000], **shape)
    for m in range(1, wl.N):
        q[:, m * wl.Hq:(m + 1) * wl.Hq] = q[:, :wl.Hq]
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, return_lse=True)
    for m in range(1, wl.N):
        assert torch.equal(out[:, m * wl.Hq:(m + 1) * wl.Hq], out[:, :wl.Hq])
        assert torch.equal(lse[:, m * wl.Hq:(m + 1) * wl.Hq], lse[:, :wl.Hq])


def test_page_permutation_gives_identical_bits():
    wl, q, k, v, pool = setup([700, 3000, 64, 9000], **LLAMA)
    out1 = pool.decode_attention(bits_to_torch(q), wl.N)
    perm = np.random.default_rng(5).permutation(wl.num_pages)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    wl2 = W.Workload(**{**wl.__dict__})
    wl2.block_table = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    pool2 = make_pool(wl2, k2, v2)
    out2 = pool2.decode_attention(bits_to_torch(q), wl.N)
    assert torch.equal(out1, out2)


def test_single_key_returns_v_exactly():
    wl, q, k, v, pool = setup([1, 1, 1], N=3, Hq=8, Hkv=2, D=128, P=16)
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    got = torch_to_bits(out)
    for b in range(wl.B):
        page = wl.block_table[b, 0]
        for r in range(wl.rows):
            np.testing.assert_array_equal(got[b, r], v[page, (r % wl.Hq) // wl.G, 0])


def test_equal_scores_return_mean_of_values():
    lens = [5, 16, 100, 1234]
    wl, q, k, v, pool = setup(lens, N=2, Hq=8, Hkv=2, D=64, P=32)
    q[:] = 0
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, return_lse=True)
    vf = W.f32_from_bf16_bits(v).astype(np.float64)
    for b, L in enumerate(lens):
        t = np.arange(L)
        vb = vf[wl.block_table[b, t // wl.P], :, t % wl.P, :]          # [L, Hkv, D]
        ref = np.stack([vb[:, (r % wl.Hq) // wl.G].mean(0) for r in range(wl.rows)])
        compare(out[b], ref, what=f"mean b={b}")
        np.testing.assert_allclose(lse[b].cpu().numpy(), np.log(L), atol=1e-4)


@pytest.mark.parametrize("shape,exact", [(LLAMA, True), (QWEN14, False)])
def test_shared_equals_unshared_per_model_runs(shape, exact):
    """Stacking decoders changes traffic, not values: slice m of the shared
    call equals a one-decoder call on model m's queries (bit-exact where both
    launches use the same warp split, within tolerance otherwise)."""
    wl, q, k, v, pool = setup([700, 3000, 64, 9000], **shape)
    qt = bits_to_torch(q)
    shared = pool.decode_attention(qt, wl.N)
    for m in range(wl.N):
        qm = qt[:, m * wl.Hq:(m + 1) * wl.Hq].contiguous()
        single = pool.decode_attention(qm, 1)
        if exact:
            assert torch.equal(shared[:, m * wl.Hq:(m + 1) * wl.Hq], single)
        else:
            compare(shared[:, m * wl.Hq:(m + 1) * wl.Hq], single.double().cpu().numpy(), what=f"m={m}")


# --------------------------------------------------------------------------
# error reporting
# --------------------------------------------------------------------------
def test_out_of_range_page_sets_flag_and_is_skipped():
    """A block-table entry outside the pool is caught by the kernel's bounds
    check before any copy: the page is skipped, SHKV_ERRF_PAGE_OOB is set and
    the other requests are unaffected."""
    wl, q, k, v, pool = setup([300, 300], **LLAMA)
    ref = pool.decode_attention(bits_to_torch(q), wl.N).clone()
    assert pool.check_errors() == 0
    pool.block_table[1, 3] = wl.num_pages + 7
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    flags = pool.check_errors()
    assert flags & N.SHKV_ERRF_PAGE_OOB
    assert torch.equal(out[0], ref[0])
    assert bool(torch.isfinite(out.float()).all())
    assert pool.check_errors() == 0          # reading clears the word


def test_a_stalled_wait_ends_with_the_timeout_flag():
    """The library's waits are bounded: a kernel whose wait nothing completes
    gives up after the limit (2 s of device time), sets SHKV_ERRF_TIMEOUT and
    exits.  The host reads the bit, and the same context then decodes the
    same bits as before."""
    import time
    wl, q, k, v, pool = setup([300, 2000], **LLAMA)
    ref = pool.decode_attention(bits_to_torch(q), wl.N).clone()
    assert pool.check_errors() == 0
    t0 = time.perf_counter()
    N.shkv_selftest_bounded_wait(pool.handle, None)
    flags = pool.check_errors()
    waited = time.perf_counter() - t0
    assert flags == N.SHKV_ERRF_TIMEOUT
    assert 1.9 < waited < 60.0
    assert pool.check_errors() == 0
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    assert pool.check_errors() == 0
    assert torch.equal(out, ref)


def test_device_length_disagreeing_with_host_copy_sets_flag():
    wl, q, k, v, pool = setup([300, 300], **LLAMA)
    pool.seq_lens[0] = 17                     # behind the pool's back
    out = pool.decode_attention(bits_to_torch(q), wl.N)
    assert pool.check_errors() & N.SHKV_ERRF_SEQ_LEN
    assert bool(torch.isfinite(out.float()).all())


def test_append_to_out_of_range_page_sets_flag():
    wl = W.custom_workload("app", B=2, N=1, Hq=2, Hkv=2, D=64, P=16, lens_prefill=[3, 3], n_append=5, seed=1)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v, lens=wl.lens_prefill)
    pool.block_table[1, 0] = -5
    kn, vn = W.gen_append(wl)
    pool.append_kv(bits_to_torch(kn), bits_to_torch(vn))
    assert pool.check_errors() & N.SHKV_ERRF_PAGE_OOB
    np.testing.assert_array_equal(torch_to_bits(pool.k_pages)[wl.block_table[0, 0], :, 3:8], kn[0].transpose(1, 0, 2))


def test_host_argument_errors():
    wl, q, k, v, pool = setup([50, 60], **LLAMA)
    qt = bits_to_torch(q)
    with pytest.raises(N.ShkvError) as e:
        pool.set_seq_lens([50, 0])
        pool.decode_attention(qt, wl.N)
    assert e.value.status == N.SHKV_ERR_INVALID_ARG
    pool.set_seq_lens([50, 60])
    with pytest.raises(N.ShkvError) as e:            # 8 decoders x 4 = 32 rows is fine; 17 x 4 > 64 is not
        big = torch.zeros((2, 17 * 32, 128), dtype=torch.bfloat16, device="cuda")
        pool.decode_attention(big, 17)
    assert e.value.status == N.SHKV_ERR_UNSUPPORTED
    with pytest.raises(N.ShkvError) as e:
        kn = torch.zeros((2, 10_000, 8, 128), dtype=torch.bfloat16, device="cuda")
        pool.append_kv(kn, kn)
    assert e.value.status == N.SHKV_ERR_CAPACITY
    with pytest.raises(N.ShkvError) as e:
        pool.set_seq_lens([50, wl.max_pages_per_seq * wl.P + 1])
    assert e.value.status == N.SHKV_ERR_CAPACITY
    assert pool.check_errors() == 0


def test_one_workspace_serves_calls_of_any_shape():
    """Decodes of different batch sizes and stacked-row counts share one
    workspace, back to back: every call's arrival counters sit in the fixed
    counter region that nothing else writes, so a call never starts from
    counters another call's partials left behind, and each matches the
    oracle."""
    import oracle
    rng = np.random.default_rng(23)
    cases = [setup([300, 2049, 64, 5000], seed=31, **LLAMA),
             setup([int(x) for x in rng.integers(1, 6000, size=40)], seed=32, **QWEN14),
             setup([9000, 17, 4000], seed=33, N=4, Hq=32, Hkv=8, D=128, P=16)]
    need = 0
    for wl, q, k, v, pool in cases:
        need = max(need, N.shkv_decode_workspace_size(pool.handle, wl.B, wl.N, wl.Hq))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    qts = [bits_to_torch(c[1]) for c in cases]
    order = [0, 1, 2, 0, 2, 1, 1, 0]
    runs = []
    for c in order:
        wl = cases[c][0]
        runs.append((c, torch.empty_like(qts[c]), torch.empty((wl.B, wl.N * wl.Hq), dtype=torch.float32,
                                                              device="cuda")))
    torch.cuda.synchronize()
    for c, out, lse in runs:
        wl, pool = cases[c][0], cases[c][4]
        N.shkv_decode_attention(pool.handle, wl.B, wl.N, wl.Hq, qts[c].data_ptr(), float(wl.scale), out.data_ptr(),
                                lse.data_ptr(), ws.data_ptr(), ws.numel(), None)
    torch.cuda.synchronize()
    refs = []
    for wl, q, k, v, pool in cases:
        assert pool.check_errors() == 0
        refs.append(oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                            scale=wl.scale))
    for i, (c, out, lse) in enumerate(runs):
        compare(out, refs[c][0], lse, refs[c][1], what=f"call {i}")
    counters = ws[: N.SHKV_COUNT_REGION_BYTES].view(torch.int32)
    assert int(counters.abs().sum()) == 0          # the counter region is left zeroed
