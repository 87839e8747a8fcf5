"""GPU parity: libshkv's CUDA path against the fp64 oracle, element by
element, on seeded inputs (all through the C ABI via the ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import (bits_to_torch, compare, make_pool, oracle_for_requests, torch_to_bits)

pytestmark = pytest.mark.gpu


def run_full(wl, q, k, v, return_lse=True):
    pool = make_pool(wl, k, v)
    qt = bits_to_torch(q)
    out, lse = pool.decode_attention(qt, wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N,
                                        hq=wl.Hq, scale=wl.scale)
    compare(out, ref, lse, lref, what=wl.name)
    return pool, out, lse


def test_tiny_config_matches_oracle():
    wl = W.make_workload("tiny")
    run_full(wl, W.gen_q(wl), *W.gen_pool(wl))


# Reduced-size versions of every configured shape: same heads, head dim,
# page size and decoder count; ragged lengths spanning many pages.
SHAPES = {
    "llama8b": dict(N=2, Hq=32, Hkv=8, D=128, P=16),
    "qwen8b": dict(N=4, Hq=32, Hkv=8, D=128, P=16),
    "qwen14b": dict(N=8, Hq=40, Hkv=8, D=128, P=32),
    "long": dict(N=8, Hq=16, Hkv=8, D=128, P=16),
    "tiny": dict(N=2, Hq=8, Hkv=2, D=64, P=16),
    "d64_p32_r16": dict(N=4, Hq=8, Hkv=2, D=64, P=32),
    "mha_n1": dict(N=1, Hq=8, Hkv=8, D=128, P=16),        # R = 1
    "r64": dict(N=8, Hq=16, Hkv=2, D=128, P=16),          # R = 64, four row groups
    "r24": dict(N=3, Hq=64, Hkv=8, D=64, P=32),           # R = 24, two row groups
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_reduced_shapes_match_oracle(shape):
    lens = [1, 15, 16, 17, 33, 257, 1000, 2049, 4100]
    wl = W.custom_workload(shape, B=len(lens), lens_prefill=lens, seed=17, **SHAPES[shape])
    run_full(wl, W.gen_q(wl), *W.gen_pool(wl))


@pytest.mark.parametrize("shape", ["llama8b", "qwen8b"])
def test_max_batch_matches_oracle(shape):
    """The largest batch one call takes (SHKV_MAX_BATCH = 1024 requests) with
    ragged short lengths: every entry of the plan's per-request tables is used
    and each CTA crosses many (request, head) units.  llama8b heads run the
    mma.sync consumer, qwen8b heads the tcgen05 one."""
    rng = np.random.default_rng(23)
    lens = rng.integers(1, 97, size=1024).tolist()
    wl = W.custom_workload(f"maxbatch_{shape}", B=len(lens), lens_prefill=lens, seed=29, **SHAPES[shape])
    run_full(wl, W.gen_q(wl), *W.gen_pool(wl))


def test_single_long_request_is_split_and_merged():
    """One request, one KV head: the whole grid works on it, so it is cut
    into many pieces that the last arriving CTA merges."""
    wl = W.custom_workload("split", B=1, N=4, Hq=4, Hkv=1, D=128, P=16, lens_prefill=[40000], seed=3)
    run_full(wl, W.gen_q(wl), *W.gen_pool(wl))


def test_repeated_calls_reuse_the_workspace():
    """The workspace's arrival counters return to zero after each call, so a
    second call on the same workspace gives the same bits."""
    wl = W.custom_workload("rep", B=3, N=2, Hq=8, Hkv=2, D=128, P=16, lens_prefill=[30000, 9000, 77], seed=5)
    q = W.gen_q(wl)
    pool, out1, lse1 = run_full(wl, q, *W.gen_pool(wl))
    out2, lse2 = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    ws = pool._workspace
    count_bytes = ((wl.B * wl.Hkv * 4 + 255) // 256) * 256
    assert int(ws[:count_bytes].count_nonzero()) == 0


def test_llama8b_full_size_matches_oracle():
    """The Llama-3.1-8B configuration at full size, every output checked."""
    wl = W.make_workload("llama8b")
    q = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl)
    pool = make_pool(wl, k_dev, v_dev)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    k, v = torch_to_bits(k_dev), torch_to_bits(v_dev)
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N,
                                        hq=wl.Hq, scale=wl.scale)
    compare(out, ref, lse, lref, what="llama8b")


def _sampled_check(name, n_sample=3):
    wl = W.make_workload(name)
    q = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl)
    pool = make_pool(wl, k_dev, v_dev)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    assert bool(torch.isfinite(out.float()).all())
    order = np.argsort(wl.lens_final)
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})[:n_sample]
    refs = oracle_for_requests(wl, q, k_dev, v_dev, picks)
    for b, (ref, lref) in refs.items():
        compare(out[b], ref, lse[b], lref, what=f"{name}[b={b}, L={wl.lens_final[b]}]")
    return wl, pool, q, out


@pytest.mark.parametrize("name", ["qwen8b", "qwen14b"])
def test_full_size_sampled_requests_match_oracle(name):
    """Full-size pools generated on the device; the shortest, median and
    longest requests are recomputed by the oracle from pages read back."""
    _sampled_check(name)


def test_long_context_with_partial_prefill_append():
    """Qwen3-1.7B shape, 4 x 131072 cached tokens plus a 512-token partial
    prefill appended through shkv_append_kv (PrefillShare Sec. 3.3), then
    decode over 131584 tokens.  The append is checked bit-exactly against the
    oracle's append on the read-back pages; decode against the oracle on two
    requests."""
    wl = W.make_workload("long")
    q = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl)
    pool = make_pool(wl, k_dev, v_dev, lens=wl.lens_prefill)
    g = torch.Generator(device="cuda").manual_seed(404)
    shape = (wl.B, wl.n_append, wl.Hkv, wl.D)
    kn = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    # pages the append touches, before
    first = [int(wl.lens_prefill[b]) // wl.P for b in range(wl.B)]
    last = [(int(wl.lens_prefill[b]) + wl.n_append - 1) // wl.P for b in range(wl.B)]
    touched = sorted({int(wl.block_table[b, pi]) for b in range(wl.B) for pi in range(first[b], last[b] + 1)})
    tt = torch.tensor(touched, device="cuda")
    k_before = torch_to_bits(k_dev.index_select(0, tt))
    v_before = torch_to_bits(v_dev.index_select(0, tt))
    pool.append_kv(kn, vn)
    assert pool.check_errors() == 0
    assert (pool.host_seq_lens(wl.B) == wl.lens_final).all()
    assert (pool.seq_lens[: wl.B].cpu().numpy() == wl.lens_final).all()
    # oracle append on a compact pool holding just the touched pages
    remap = {p: i for i, p in enumerate(touched)}
    bt_small = np.full_like(wl.block_table, -1)
    for b in range(wl.B):
        for pi in range(first[b], last[b] + 1):
            bt_small[b, pi] = remap[int(wl.block_table[b, pi])]
    k_exp, v_exp, lens_exp = oracle.append_kv(k_before, v_before, bt_small, wl.lens_prefill,
                                              torch_to_bits(kn), torch_to_bits(vn))
    np.testing.assert_array_equal(torch_to_bits(k_dev.index_select(0, tt)), k_exp)
    np.testing.assert_array_equal(torch_to_bits(v_dev.index_select(0, tt)), v_exp)
    np.testing.assert_array_equal(lens_exp, wl.lens_final)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    refs = oracle_for_requests(wl, q, k_dev, v_dev, [0, 3])
    for b, (ref, lref) in refs.items():
        compare(out[b], ref, lse[b], lref, what=f"long[b={b}]")


def test_append_small_matches_oracle_bit_exactly():
    wl = W.custom_workload("app", B=5, N=2, Hq=8, Hkv=2, D=64, P=16,
                           lens_prefill=[1, 15, 16, 40, 100], n_append=37, seed=8)
    k, v = W.gen_pool(wl)
    kn, vn = W.gen_append(wl)
    pool = make_pool(wl, k, v, lens=wl.lens_prefill)
    pool.append_kv(bits_to_torch(kn), bits_to_torch(vn))
    assert pool.check_errors() == 0
    k_exp, v_exp, lens_exp = oracle.append_kv(k, v, wl.block_table, wl.lens_prefill, kn, vn)
    np.testing.assert_array_equal(torch_to_bits(pool.k_pages), k_exp)
    np.testing.assert_array_equal(torch_to_bits(pool.v_pages), v_exp)
    np.testing.assert_array_equal(pool.seq_lens[: wl.B].cpu().numpy(), lens_exp)
    # and decode over the extended cache
    q = W.gen_q(wl)
    out, lse = pool.decode_attention(bits_to_torch(q), wl.N, scale=wl.scale, return_lse=True)
    ref, lref = oracle.decode_attention(q, k_exp, v_exp, wl.block_table, lens_exp, n_models=wl.N,
                                        hq=wl.Hq, scale=wl.scale)
    compare(out, ref, lse, lref, what="append+decode")


def test_splitkv_merge_matches_oracle():
    rng = np.random.default_rng(0)
    S, B, rows, D = 7, 3, 10, 128
    o = rng.standard_normal((S, B, rows, D))
    l = rng.standard_normal((S, B, rows)) * 3
    l[2, 0, :] = -np.inf                 # a split with no tokens
    l[:, 1, 3] = -np.inf                 # a row with no tokens at all
    from cross_model_shared_gb300 import splitkv_merge
    out, lse = splitkv_merge(torch.from_numpy(o.astype(np.float32)).cuda(),
                             torch.from_numpy(l.astype(np.float32)).cuda())
    torch.cuda.synchronize()
    ref, lref = oracle.splitkv_merge(o.astype(np.float32).astype(np.float64),
                                     l.astype(np.float32).astype(np.float64))
    compare(out, ref, what="merge")
    lg = lse.cpu().numpy()
    assert np.isneginf(lg[1, 3]) and np.isneginf(lref[1, 3])
    fin = np.isfinite(lref)
    assert np.abs(lg[fin] - lref[fin]).max() <= 1e-5 * max(1.0, np.abs(lref[fin]).max())
