"""Pins for the oracle's per-decoder unique tails (PrefillShare Sec. 3.3-4,
Eqs. 8-9: decode starts from the shared base cache and each decoder extends
it with its own generated-token cache; decoder m attends the concatenation
of the shared prefix and its own tail).

Each pin checks the oracle against something other than itself: the
shared-only oracle when every tail is empty, a numpy/scipy brute force over
the explicit concatenation, the invariance of moving shared tokens into
every tail, and closed forms.
"""
import numpy as np
import pytest
import scipy.special

import oracle
from cross_model_shared_gb300 import workloads as W


def widen(bits):
    return W.f32_from_bf16_bits(bits).astype(np.float64)


def setup(lens, tail_lens, N=3, Hq=4, Hkv=2, D=64, P=16, seed=11):
    tail_lens = np.asarray(tail_lens).reshape(len(lens), N)
    wl = W.custom_workload("tails", B=len(lens), N=N, Hq=Hq, Hkv=Hkv, D=D, P=P, lens_prefill=lens, seed=seed,
                           spare_pages=W.tails_spare_pages(tail_lens, P) + 3)
    tt, tl = W.make_tails(wl, tail_lens, seed=seed + 1)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    return wl, tt, tl, q, k, v


def run(wl, tt, tl, q, k, v):
    return oracle.decode_attention_tails(q, k, v, wl.block_table, wl.lens_final, tt, tl, n_models=wl.N,
                                         hq=wl.Hq, scale=wl.scale)


def concat_tokens(pool, wl, tt, tl, b, m):
    """[L_b + T_bm, Hkv, D] by numpy indexing: shared prefix, then the tail."""
    P = wl.P
    L = int(wl.lens_final[b])
    T = int(tl[b, m])
    t = np.arange(L)
    shared = pool[wl.block_table[b, t // P], :, t % P, :]
    u = np.arange(T)
    tail = pool[tt[b, m, u // P], :, u % P, :]
    return np.concatenate([shared, tail], axis=0)


def test_empty_tails_equal_the_shared_only_oracle():
    """With every tail empty the concatenation is the shared prefix: the
    result is the shared-only oracle's, bit for bit (same tokens, same order,
    same fp64 operations)."""
    lens = [5, 40, 17]
    wl, tt, tl, q, k, v = setup(lens, np.zeros((3, 3), int))
    out, lse = run(wl, tt, tl, q, k, v)
    ref, lref = oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                        scale=wl.scale)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, lref)


def test_brute_force_over_the_concatenation():
    """Textbook softmax (scipy) on a numpy gather of [shared ++ tail of
    decoder m]: pins the per-decoder tail selection, the tail page walk, the
    tail-length mask and the GQA head map."""
    lens = [9, 33, 1, 20]
    tails = [[0, 5, 17], [16, 1, 0], [3, 40, 2], [0, 0, 31]]
    wl, tt, tl, q, k, v = setup(lens, tails)
    out, lse = run(wl, tt, tl, q, k, v)
    for b in range(wl.B):
        for m in range(wl.N):
            kb = widen(concat_tokens(k, wl, tt, tl, b, m))
            vb = widen(concat_tokens(v, wl, tt, tl, b, m))
            for h in range(wl.Hq):
                r = m * wl.Hq + h
                g = h // wl.G
                s = wl.scale * kb[:, g] @ widen(q[b, r])
                np.testing.assert_allclose(out[b, r], scipy.special.softmax(s) @ vb[:, g], rtol=0, atol=1e-12)
                assert lse[b, r] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


def test_moving_shared_tokens_into_every_tail_changes_nothing():
    """Attention depends on the concatenated token list only: shortening the
    shared prefix by k tokens and prepending those same tokens (copied to
    fresh pages) to every decoder's tail gives the same result."""
    lens = [40, 25]
    tails = [[7, 0, 3], [12, 30, 1]]
    wl, tt, tl, q, k, v = setup(lens, tails, P=16)
    out, lse = run(wl, tt, tl, q, k, v)
    kcut = 16                                   # one whole page of every request
    lens2 = (wl.lens_final - kcut).astype(np.int32)
    # new tails: [the cut shared page] ++ old tail, rebuilt page by page in fresh pool pages
    P = wl.P
    new_lens = tl + kcut
    width = int(((new_lens + P - 1) // P).max())
    extra = int(((new_lens + P - 1) // P).sum())
    k2 = np.concatenate([k, np.zeros((extra,) + k.shape[1:], k.dtype)])
    v2 = np.concatenate([v, np.zeros((extra,) + v.shape[1:], v.dtype)])
    tt2 = np.full((wl.B, wl.N, width), -1, np.int32)
    nxt = k.shape[0]
    for b in range(wl.B):
        # the cut tokens are the last kcut shared tokens: positions L-kcut .. L-1
        L = int(wl.lens_final[b])
        t = np.arange(L - kcut, L)
        cut_k = k[wl.block_table[b, t // P], :, t % P, :]
        cut_v = v[wl.block_table[b, t // P], :, t % P, :]
        for m in range(wl.N):
            T = int(tl[b, m])
            u = np.arange(T)
            seq_k = np.concatenate([cut_k, k[tt[b, m, u // P], :, u % P, :]])
            seq_v = np.concatenate([cut_v, v[tt[b, m, u // P], :, u % P, :]])
            n = len(seq_k)
            for pi in range((n + P - 1) // P):
                rows = slice(pi * P, min(n, (pi + 1) * P))
                cnt = rows.stop - rows.start
                k2[nxt, :, :cnt] = seq_k[rows].transpose(1, 0, 2)
                v2[nxt, :, :cnt] = seq_v[rows].transpose(1, 0, 2)
                tt2[b, m, pi] = nxt
                nxt += 1
    out2, lse2 = oracle.decode_attention_tails(q, k2, v2, wl.block_table, lens2, tt2,
                                               new_lens.astype(np.int32), n_models=wl.N, hq=wl.Hq, scale=wl.scale)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


def test_identical_queries_and_tails_give_identical_slices_and_distinct_tails_differ():
    """Decoders with identical queries and identical tails get identical
    slices; giving one decoder a different tail changes its slice only."""
    lens = [30, 12]
    wl, tt, tl, q, k, v = setup(lens, [[6, 6, 6], [9, 9, 9]])
    for m in range(1, wl.N):
        q[:, m * wl.Hq:(m + 1) * wl.Hq] = q[:, :wl.Hq]
        tt[:, m] = tt[:, 0]
    out, lse = run(wl, tt, tl, q, k, v)
    for m in range(1, wl.N):
        np.testing.assert_array_equal(out[:, m * wl.Hq:(m + 1) * wl.Hq], out[:, :wl.Hq])
    tl2 = tl.copy()
    tl2[:, 2] -= 3
    out2, _ = run(wl, tt, tl2, q, k, v)
    np.testing.assert_array_equal(out2[:, :2 * wl.Hq], out[:, :2 * wl.Hq])
    assert np.abs(out2[:, 2 * wl.Hq:] - out[:, 2 * wl.Hq:]).max() > 1e-3


def test_dominant_tail_token_returns_its_value():
    """One tail token whose key is a large multiple of the query takes all
    the softmax mass: the row returns that token's V (to exp(-huge) ~ 0)."""
    lens = [10]
    wl, tt, tl, q, k, v = setup(lens, [[4, 4, 4]], N=3, Hq=2, Hkv=1)
    P = wl.P
    for m in range(wl.N):
        page, slot = tt[0, m, 2 // P], 2 % P          # tail token 2 of decoder m
        qm = widen(q[0, m * wl.Hq])
        k[page, 0, slot] = W.bf16_bits_from_f32((qm * 64.0).astype(np.float32))
        q[0, m * wl.Hq + 1] = q[0, m * wl.Hq]
    out, _ = run(wl, tt, tl, q, k, v)
    for m in range(wl.N):
        page, slot = tt[0, m, 2 // P], 2 % P
        np.testing.assert_allclose(out[0, m * wl.Hq], widen(v[page, 0, slot]), rtol=0, atol=1e-9)
