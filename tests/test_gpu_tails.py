"""Per-decoder unique tails on the GPU against the fp64 oracle.

Decoder m of request b attends the shared prefix and its own tail
(PrefillShare Sec. 3.3-4, Eqs. 8-9).  The library streams each request's
shared pages and then every decoder's tail pages in one pass, a tail page
attended by its own decoder's rows only; these tests compare with the
oracle's direct definition over the concatenated token list.
"""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import DecoderTails
from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, make_pool, torch_to_bits

pytestmark = pytest.mark.gpu

SHAPES = {
    "llama8b": dict(N=2, Hq=32, Hkv=8, D=128, P=16),      # shared pass R = 8 (mma.sync)
    "qwen14b": dict(N=8, Hq=40, Hkv=8, D=128, P=32),      # shared pass R = 40 (tcgen05)
    "qwen8b": dict(N=4, Hq=32, Hkv=8, D=128, P=16),       # R = 16: tcgen05 with 16-token pages (two producers)
    "d64": dict(N=3, Hq=8, Hkv=2, D=64, P=16),            # head dim 64
    "r8_p32": dict(N=2, Hq=32, Hkv=8, D=128, P=32),       # R = 8 (mma.sync) with one 32-token page a stage
}


def setup(shape, lens, tails, seed=5, reserve_tokens=0):
    sh = SHAPES[shape]
    tails = np.asarray(tails).reshape(len(lens), sh["N"])
    spare = W.tails_spare_pages(tails, sh["P"], reserve_tokens)
    wl = W.custom_workload(shape, B=len(lens), lens_prefill=lens, seed=seed, spare_pages=spare, **sh)
    tt, tl = W.make_tails(wl, tails, seed=seed + 1, reserve_tokens=reserve_tokens, extra_pages_per_tail=1)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    tails_obj = DecoderTails(pool, wl.B, wl.N, tt.shape[2], initial_tail_lens=tl)
    tails_obj.block_table.copy_(torch.from_numpy(tt))
    torch.cuda.synchronize()
    return wl, tt, tl, q, k, v, pool, tails_obj


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_tails_match_oracle(shape):
    lens = [1, 17, 300, 2049, 64]
    rng = np.random.default_rng(3)
    tails = rng.integers(0, 400, size=(len(lens), SHAPES[shape]["N"]))
    tails[0, 0] = 0
    tails[1, :] = 0
    tails[2, -1] = 1
    wl, tt, tl, q, k, v, pool, tob = setup(shape, lens, tails)
    out, lse = tob.decode_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention_tails(q, k, v, wl.block_table, wl.lens_final, tt, tl, n_models=wl.N,
                                              hq=wl.Hq, scale=wl.scale)
    compare(out, ref, lse, lref, what=f"tails {shape}")


@pytest.mark.parametrize("shape", ["llama8b", "qwen14b", "r8_p32"])
def test_empty_tails_give_the_plain_decode_bits(shape):
    """Every tail empty: the merge has one live split with weight exactly 1,
    so the result is the shared decode's own bits."""
    lens = [5, 300, 2049]
    wl, tt, tl, q, k, v, pool, tob = setup(shape, lens, np.zeros((3, SHAPES[shape]["N"]), int))
    qt = bits_to_torch(q)
    out_t, lse_t = tob.decode_attention(qt, scale=wl.scale, return_lse=True)
    out_p, lse_p = pool.decode_attention(qt, wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    assert torch.equal(out_t, out_p)
    assert torch.equal(lse_t, lse_p)


def test_long_tails_are_split_and_merged():
    """Tails long enough that the tail pass itself splits across CTAs."""
    lens = [3000]
    wl, tt, tl, q, k, v, pool, tob = setup("qwen14b", lens, [[9000, 1, 0, 4000, 20000, 33, 7, 128]])
    out, lse = tob.decode_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention_tails(q, k, v, wl.block_table, wl.lens_final, tt, tl, n_models=wl.N,
                                              hq=wl.Hq, scale=wl.scale)
    compare(out, ref, lse, lref, what="long tails")


def test_tail_append_then_decode():
    """Decoders append their own generated tokens (different K/V per
    decoder) into pre-assigned tail pages, then decode: the tails' bytes
    match numpy indexing and the result matches the oracle."""
    lens = [100, 40]
    tails0 = np.array([[3, 0], [16, 15]])
    T = 5
    wl, tt, tl, q, k, v, pool, tob = setup("llama8b", lens, tails0, reserve_tokens=T)
    rng = np.random.default_rng(9)
    kn = W.bf16_bits_from_f32(rng.standard_normal((wl.B, wl.N, T, wl.Hkv, wl.D)).astype(np.float32))
    vn = W.bf16_bits_from_f32(rng.standard_normal((wl.B, wl.N, T, wl.Hkv, wl.D)).astype(np.float32))
    tob.append(bits_to_torch(kn), bits_to_torch(vn))
    assert pool.check_errors() == 0
    np.testing.assert_array_equal(tob.host_lens(wl.B), tl + T)
    k2, v2 = torch_to_bits(pool.k_pages), torch_to_bits(pool.v_pages)
    tl2 = tl + T
    for b in range(wl.B):
        for m in range(wl.N):
            for i in range(T):
                pos = int(tl[b, m]) + i
                page, slot = tt[b, m, pos // wl.P], pos % wl.P
                np.testing.assert_array_equal(k2[page, :, slot], kn[b, m, i])
                np.testing.assert_array_equal(v2[page, :, slot], vn[b, m, i])
    out, lse = tob.decode_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.decode_attention_tails(q, k2, v2, wl.block_table, wl.lens_final, tt, tl2.astype(np.int32),
                                              n_models=wl.N, hq=wl.Hq, scale=wl.scale)
    compare(out, ref, lse, lref, what="tails after append")


def test_identical_tails_and_queries_give_matching_slices():
    """Decoders with identical queries and identical tails get the same
    result; each (request, decoder) tail is its own unit of the split plan,
    so equal tails may be split differently: equal within the tolerance, not
    bit for bit."""
    lens = [700, 64]
    wl, tt, tl, q, k, v, pool, tob = setup("qwen14b", lens, [[50] * 8, [200] * 8])
    for m in range(1, wl.N):
        q[:, m * wl.Hq:(m + 1) * wl.Hq] = q[:, :wl.Hq]
    tt2 = tt.copy()
    tt2[:, 1:] = tt[:, :1]
    tob.block_table.copy_(torch.from_numpy(tt2))
    out = tob.decode_attention(bits_to_torch(q), scale=wl.scale)
    first = out[:, :wl.Hq].double().cpu().numpy()
    for m in range(1, wl.N):
        compare(out[:, m * wl.Hq:(m + 1) * wl.Hq], first, what=f"decoder {m} vs 0")


def test_out_of_range_tail_page_sets_flag():
    lens = [100, 100]
    wl, tt, tl, q, k, v, pool, tob = setup("llama8b", lens, [[40, 40], [40, 40]])
    tob.block_table[1, 1, 0] = wl.num_pages + 3
    out = tob.decode_attention(bits_to_torch(q), scale=wl.scale)
    assert pool.check_errors() & N.SHKV_ERRF_PAGE_OOB
    assert bool(torch.isfinite(out.float()).all())


@pytest.mark.parametrize("name", ["llama8b", "qwen8b"])
def test_full_size_tails_sampled_requests(name):
    """A full-size workload with 128-384-token tails per decoder (pools on the
    device); the shortest, median and longest requests are recomputed by the
    oracle from their shared and tail pages read back."""
    base = W.make_workload(name)
    rng = np.random.default_rng(base.seed + 4242)
    tails = rng.integers(128, 385, size=(base.B, base.N)).astype(np.int32)
    wl = W.custom_workload(f"{name}+tails", B=base.B, N=base.N, Hq=base.Hq, Hkv=base.Hkv, D=base.D, P=base.P,
                           lens_prefill=base.lens_prefill, n_append=base.n_append, seed=base.seed,
                           spare_pages=W.tails_spare_pages(tails, base.P))
    tt, tl = W.make_tails(wl, tails, seed=wl.seed + 1)
    q = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl)
    pool = make_pool(wl, k_dev, v_dev)
    tob = DecoderTails(pool, wl.B, wl.N, tt.shape[2], initial_tail_lens=tl)
    tob.block_table.copy_(torch.from_numpy(tt))
    out, lse = tob.decode_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    assert bool(torch.isfinite(out.float()).all())
    order = np.argsort(wl.lens_final)
    for b in sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])}):
        npg = int((wl.lens_final[b] + wl.P - 1) // wl.P)
        tpg = [int((tl[b, m] + wl.P - 1) // wl.P) for m in range(wl.N)]
        ids = np.concatenate([wl.block_table[b, :npg]] + [tt[b, m, :tpg[m]] for m in range(wl.N)]).astype(np.int64)
        sel = torch.from_numpy(ids).to(k_dev.device)
        kb, vb = torch_to_bits(k_dev.index_select(0, sel)), torch_to_bits(v_dev.index_select(0, sel))
        # the request's pages renumbered 0.. in the order gathered: shared, then each tail
        bt = np.arange(npg, dtype=np.int32)[None, :]
        ttb = np.full((1, wl.N, max(1, max(tpg))), -1, np.int32)
        off = npg
        for m in range(wl.N):
            ttb[0, m, :tpg[m]] = np.arange(off, off + tpg[m], dtype=np.int32)
            off += tpg[m]
        ref, lref = oracle.decode_attention_tails(q[b:b + 1], kb, vb, bt, np.array([wl.lens_final[b]], np.int32),
                                                  ttb, tl[b:b + 1], n_models=wl.N, hq=wl.Hq, scale=wl.scale)
        compare(out[b], ref[0], lse[b], lref[0], what=f"{name}+tails[b={b}, L={wl.lens_final[b]}]")


@pytest.mark.parametrize("shape", ["qwen8b", "llama8b"])
def test_back_to_back_calls_on_one_workspace(shape):
    """A call's unit-layout kernel runs while the previous call's decode is
    still running, writing its tables where the previous call's are not (or
    waiting first when shapes leave no such place).  Calls that cycle through
    three pools of different shapes (batch, strides, so different table
    positions) on one shared workspace, enqueued with no synchronisation
    between them, each give their own oracle result."""
    rng = np.random.default_rng(17)
    n = SHAPES[shape]["N"]
    cases = [setup(shape, [300, 2049, 64, 5000], rng.integers(0, 400, size=(4, n)), seed=5),
             setup(shape, [4000, 17, 900], rng.integers(0, 700, size=(3, n)), seed=9),
             setup(shape, [int(x) for x in rng.integers(1, 3000, size=12)], rng.integers(0, 1500, size=(12, n)),
                   seed=11)]
    order = [0, 1, 0, 2, 1, 2, 0, 0, 2, 2, 1, 0]
    need = 0
    for wl, tt, tl, q, k, v, pool, tob in cases:
        need = max(need, N.shkv_decode_tails_workspace_size(pool.handle, tob.handle, wl.B, wl.Hq))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    qts = [bits_to_torch(c[3]) for c in cases]
    runs = []
    for c in order:
        wl = cases[c][0]
        out = torch.empty_like(qts[c])
        lse = torch.empty((wl.B, wl.N * wl.Hq), dtype=torch.float32, device="cuda")
        runs.append((c, out, lse))
    torch.cuda.synchronize()
    for c, out, lse in runs:            # twelve calls back to back, nothing between them
        wl, pool, tob = cases[c][0], cases[c][6], cases[c][7]
        N.shkv_decode_attention_tails(pool.handle, tob.handle, wl.B, wl.Hq, qts[c].data_ptr(), float(wl.scale),
                                      out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), None)
    torch.cuda.synchronize()
    refs = []
    for wl, tt, tl, q, k, v, pool, tob in cases:
        assert pool.check_errors() == 0
        refs.append(oracle.decode_attention_tails(q, k, v, wl.block_table, wl.lens_final, tt, tl, n_models=wl.N,
                                                  hq=wl.Hq, scale=wl.scale))
    for i, (c, out, lse) in enumerate(runs):
        compare(out, refs[c][0], lse, refs[c][1], what=f"call {i}")
    for c in range(len(cases)):     # every call of a case gives the same bits
        same = [r for r in runs if r[0] == c]
        assert all(torch.equal(r[1], same[0][1]) and torch.equal(r[2], same[0][2]) for r in same)


@pytest.mark.parametrize("shape", ["qwen8b", "llama8b"])
def test_next_call_workspace_over_the_running_calls_workspace(shape):
    """Stream order lets a call use, as its workspace, bytes that the previous
    call is still using under another pointer, so long as its own counter
    region starts zeroed.  Here call B's workspace starts below call A's, so
    that B's first table position is A's counter region, while A's decode is
    still running when B's unit-layout kernel starts.  That kernel writes
    before waiting, so it must find a position clear of every byte A's
    kernels touch (or wait): both calls give the bits they give alone."""
    rng = np.random.default_rng(29)
    n = SHAPES[shape]["N"]
    a = setup(shape, [9000, 12000, 7000, 15000], rng.integers(0, 400, size=(4, n)), seed=5)
    b = setup(shape, [4000, 17, 900], rng.integers(0, 700, size=(3, n)), seed=9)

    def run(case, ws_ptr, ws_bytes):
        wl, pool, tob = case[0], case[6], case[7]
        qt = bits_to_torch(case[3])
        out = torch.empty_like(qt)
        lse = torch.empty((wl.B, wl.N * wl.Hq), dtype=torch.float32, device="cuda")
        N.shkv_decode_attention_tails(pool.handle, tob.handle, wl.B, wl.Hq, qt.data_ptr(), float(wl.scale),
                                      out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes, None)
        return qt, out, lse

    need = {id(c): N.shkv_decode_tails_workspace_size(c[6].handle, c[7].handle, c[0].B, c[0].Hq) for c in (a, b)}
    alone = []
    for c in (a, b):
        ws = torch.zeros(need[id(c)], dtype=torch.uint8, device="cuda")
        alone.append(run(c, ws.data_ptr(), ws.numel()))
        torch.cuda.synchronize()
    wlb = b[0]
    d_b = -(-N.shkv_decode_workspace_size(b[6].handle, wlb.B, wlb.N, wlb.Hq) // 256) * 256   # B's decode part
    a_off = d_b - 256                       # A's counters begin 256 bytes before B's first table position
    arena = torch.zeros(max(a_off + need[id(a)], need[id(b)]) + 4096, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    ra = run(a, arena.data_ptr() + a_off, need[id(a)])
    rb = run(b, arena.data_ptr(), need[id(b)])          # enqueued right behind A, nothing between them
    torch.cuda.synchronize()
    assert a[6].check_errors() == 0
    for (q0, o0, l0), (q1, o1, l1), what in ((alone[0], ra, "A"), (alone[1], rb, "B")):
        assert torch.equal(o0, o1) and torch.equal(l0, l1), what
    ref = oracle.decode_attention_tails(a[3], a[4], a[5], a[0].block_table, a[0].lens_final, a[1], a[2],
                                        n_models=a[0].N, hq=a[0].Hq, scale=a[0].scale)
    compare(ra[1], ref[0], ra[2], ref[1], what="A")
