"""Pins for the fp64 oracle, each against something other than the oracle.

The attention the oracle computes is plain softmax attention per query row
(ICaRus key design 3: the concatenated queries of N decoders attend one
shared KV; concatenation changes traffic, not values).  These tests fix it
with closed forms, invariants, library routines and hand-derived golden
values, chosen so a dropped term, a wrong index or sign, or a swapped K/V
operand fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from cross_model_shared_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def widen(bits):
    return W.f32_from_bf16_bits(bits).astype(np.float64)


def np_gather(pool, bt, b, L):
    """Logical [L, Hkv, D] view of request b by numpy fancy indexing."""
    P = pool.shape[2]
    t = np.arange(L)
    return pool[bt[b, t // P], :, t % P, :]


def small(lens, N=2, Hq=8, Hkv=2, D=64, P=16, seed=7, **kw):
    wl = W.custom_workload("pin", B=len(lens), N=N, Hq=Hq, Hkv=Hkv, D=D, P=P,
                           lens_prefill=lens, seed=seed, **kw)
    q = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    return wl, q, k, v


def run(wl, q, k, v, **kw):
    return oracle.decode_attention(q, k, v, wl.block_table, wl.lens_final, n_models=wl.N,
                                   hq=wl.Hq, scale=kw.pop("scale", wl.scale), **kw)


# --------------------------------------------------------------------------
def test_single_key_returns_its_value_and_score():
    """L=1: softmax of one score is 1, so every row returns V of its KV head
    exactly, and lse is the single scaled score.  Pins the GQA head map
    (g = h // G), V (not K) as the weighted operand, the q row index and the
    scale."""
    wl, q, k, v = small([1, 1, 1], N=2, Hq=8, Hkv=2)
    out, lse = run(wl, q, k, v)
    G = wl.G
    for b in range(wl.B):
        page = wl.block_table[b, 0]
        for m in range(wl.N):
            for h in range(wl.Hq):
                r = m * wl.Hq + h
                np.testing.assert_array_equal(out[b, r], widen(v[page, h // G, 0]))
                s = wl.scale * np.dot(widen(q[b, r]), widen(k[page, h // G, 0]))
                assert lse[b, r] == pytest.approx(s, rel=1e-13, abs=1e-13)


def test_equal_scores_return_mean_of_values():
    """q = 0 makes every score 0: out = mean of V over the L cached tokens and
    lse = ln L.  Ragged lengths with random garbage in the unused tail slots
    pin the t < L mask and the page walk."""
    lens = [37, 16, 50, 1]
    wl, q, k, v = small(lens, N=3, Hq=4, Hkv=2, D=64, P=16)
    q[:] = 0
    out, lse = run(wl, q, k, v)
    for b, L in enumerate(lens):
        vb = widen(np_gather(v, wl.block_table, b, L))      # [L, Hkv, D]
        for r in range(wl.rows):
            g = (r % wl.Hq) // wl.G
            np.testing.assert_allclose(out[b, r], vb[:, g].mean(axis=0), rtol=0, atol=1e-13)
            assert lse[b, r] == pytest.approx(math.log(L), abs=1e-13)


def test_identical_keys_return_mean_of_values():
    """All keys equal => equal scores for any query => mean of V."""
    lens = [29, 64]
    wl, q, k, v = small(lens, N=2, Hq=4, Hkv=1, D=64, P=16)
    k[:] = k[0, 0, 0]
    out, _ = run(wl, q, k, v)
    for b, L in enumerate(lens):
        vb = widen(np_gather(v, wl.block_table, b, L))
        for r in range(wl.rows):
            np.testing.assert_allclose(out[b, r], vb[:, 0].mean(axis=0), rtol=0, atol=1e-12)


def test_matches_library_softmax_attention():
    """One decoder, one query head per KV head: each row is textbook
    softmax(q K^T * scale) V over the request's tokens, computed here with
    scipy.special.softmax / logsumexp on a numpy gather of a randomly
    permuted page layout."""
    lens = [1, 15, 16, 17, 100, 257]
    wl, q, k, v = small(lens, N=1, Hq=4, Hkv=4, D=64, P=16, seed=11)
    out, lse = run(wl, q, k, v)
    for b, L in enumerate(lens):
        kb = widen(np_gather(k, wl.block_table, b, L))
        vb = widen(np_gather(v, wl.block_table, b, L))
        for h in range(wl.Hq):
            s = wl.scale * (kb[:, h] @ widen(q[b, h]))
            ref = scipy.special.softmax(s) @ vb[:, h]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-13)
            assert lse[b, h] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


def test_scale_argument_is_applied():
    """Doubling the scale equals doubling the query (bf16 doubling is exact)."""
    lens = [33, 70]
    wl, q, k, v = small(lens, seed=5)
    out1, lse1 = run(wl, q, k, v, scale=2 * wl.scale)
    q2 = W.bf16_bits_from_f32(2 * W.f32_from_bf16_bits(q))
    out2, lse2 = run(wl, q2, k, v)
    np.testing.assert_allclose(out1, out2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse1, lse2, rtol=0, atol=1e-12)


def test_identical_queries_across_models_give_identical_outputs():
    """ICaRus key design 2: one identical cache for all decoders, so equal
    query sets must give equal output slices."""
    wl, q, k, v = small([45, 130], N=4, Hq=8, Hkv=2)
    for m in range(1, wl.N):
        q[:, m * wl.Hq:(m + 1) * wl.Hq] = q[:, :wl.Hq]
    out, lse = run(wl, q, k, v)
    for m in range(1, wl.N):
        np.testing.assert_array_equal(out[:, m * wl.Hq:(m + 1) * wl.Hq], out[:, :wl.Hq])
        np.testing.assert_array_equal(lse[:, m * wl.Hq:(m + 1) * wl.Hq], lse[:, :wl.Hq])


def test_stacked_models_equal_single_model_runs():
    """Concatenating decoders along heads (ICaRus key design 3) must not
    change any decoder's result: slice m of the stacked call equals a
    one-decoder call on decoder m's queries.  Pins the model-major row order
    on both the query and the output side."""
    wl, q, k, v = small([19, 77, 200], N=3, Hq=8, Hkv=2, seed=3)
    out, lse = run(wl, q, k, v)
    for m in range(wl.N):
        qm = np.ascontiguousarray(q[:, m * wl.Hq:(m + 1) * wl.Hq])
        om, lm = oracle.decode_attention(qm, k, v, wl.block_table, wl.lens_final, n_models=1,
                                         hq=wl.Hq, scale=wl.scale)
        np.testing.assert_array_equal(out[:, m * wl.Hq:(m + 1) * wl.Hq], om)
        np.testing.assert_array_equal(lse[:, m * wl.Hq:(m + 1) * wl.Hq], lm)


def test_page_permutation_invariance():
    """Moving physical pages and rewriting the block table leaves the
    logical cache, hence the result, bit-identical."""
    wl, q, k, v = small([40, 90, 16], N=2, Hq=8, Hkv=2, seed=9)
    out, lse = run(wl, q, k, v)
    rng = np.random.default_rng(123)
    perm = rng.permutation(wl.num_pages)            # new slot of old page i
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    bt2 = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.decode_attention(q, k2, v2, bt2, wl.lens_final, n_models=wl.N,
                                         hq=wl.Hq, scale=wl.scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_split_merge_equals_unsplit():
    """Partials over disjoint token windows, merged by log-sum-exp, equal the
    unsplit attention (including an empty window, which carries no weight)."""
    wl, q, k, v = small([100, 33, 250], N=2, Hq=8, Hkv=2, seed=4)
    full, lse_full = run(wl, q, k, v)
    cuts = [0, 16, 48, 48, 129, 2**31 - 1]
    parts = [run(wl, q, k, v, t_begin=a, t_end=b) for a, b in zip(cuts[:-1], cuts[1:])]
    o_part = np.stack([p[0] for p in parts])
    l_part = np.stack([p[1] for p in parts])
    assert np.isneginf(l_part[2]).all()              # the empty window
    merged, lse = oracle.splitkv_merge(o_part, l_part)
    np.testing.assert_allclose(merged, full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_full, rtol=0, atol=1e-12)


def test_merge_closed_forms():
    """Equal lse => plain average and lse + ln 2; an lse = -inf partial has
    zero weight; all -inf => zero output and -inf lse."""
    rng = np.random.default_rng(0)
    o = rng.standard_normal((2, 1, 3, 8))
    l = np.array([[[0.5, -np.inf, -np.inf]], [[0.5, 1.25, -np.inf]]])
    out, lse = oracle.splitkv_merge(o, l)
    np.testing.assert_allclose(out[0, 0], 0.5 * (o[0, 0, 0] + o[1, 0, 0]), atol=1e-15)
    assert lse[0, 0] == pytest.approx(0.5 + math.log(2), abs=1e-15)
    np.testing.assert_array_equal(out[0, 1], o[1, 0, 1])
    assert lse[0, 1] == 1.25
    np.testing.assert_array_equal(out[0, 2], np.zeros(8))
    assert np.isneginf(lse[0, 2])
    # unequal weights: w = (1, e) for lse = (0, 1)
    o2 = np.stack([np.ones((1, 1, 4)), 3 * np.ones((1, 1, 4))])
    l2 = np.array([[[0.0]], [[1.0]]])
    out2, lse2 = oracle.splitkv_merge(o2, l2)
    e = math.e
    np.testing.assert_allclose(out2[0, 0], (1 + 3 * e) / (1 + e) * np.ones(4), atol=1e-15)
    assert lse2[0, 0] == pytest.approx(math.log(1 + e), abs=1e-15)


def test_golden_closed_form_examples():
    """Hand-derived examples whose results are closed forms (logistic /
    softmax of integer scores); the fixture lists the derivation."""
    cases = _read_golden(os.path.join(GOLDEN, "closed_form_attention.txt"))
    assert len(cases) >= 3
    for c in cases:
        D, L = c["D"], c["L"]
        P = 16
        kp = np.zeros((1, 1, P, D), np.uint16)
        vp = np.zeros((1, 1, P, D), np.uint16)
        kp[0, 0, :L] = W.bf16_bits_from_f32(np.array(c["K"], np.float32).reshape(L, D))
        vp[0, 0, :L] = W.bf16_bits_from_f32(np.array(c["V"], np.float32).reshape(L, D))
        q = W.bf16_bits_from_f32(np.array(c["q"], np.float32).reshape(1, 1, D))
        out, lse = oracle.decode_attention(q, kp, vp, np.zeros((1, 1), np.int32),
                                           np.array([L], np.int32), n_models=1, hq=1,
                                           scale=c["scale"])
        np.testing.assert_allclose(out[0, 0], c["out"], rtol=0, atol=1e-15)
        assert lse[0, 0] == pytest.approx(c["lse"], abs=1e-15)


def _closed_form(expr):
    """Evaluate a fixture expression over e, exp and log only."""
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "exp": math.exp, "log": math.log}))


def _read_golden(path):
    cases, cur = [], None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, val = line.partition("=")
            key, val = key.strip(), val.strip()
            if key == "case":
                cur = {"name": val}
                cases.append(cur)
            elif key in ("D", "L"):
                cur[key] = int(val)
            elif key == "scale":
                cur[key] = float(val)
            elif key == "lse":
                cur[key] = _closed_form(val)
            elif key == "out":
                cur[key] = [_closed_form(x) for x in val.split()]
            else:
                cur[key] = [float(x) for x in val.split()]
    return cases


def test_append_then_gather():
    """PrefillShare partial prefill: appended tokens land at positions
    L_b..L_b+T-1 of each request (bit copy), the rest of the pool is
    untouched, and lengths grow by T.  Checked with numpy indexing."""
    wl = W.custom_workload("app", B=3, N=1, Hq=2, Hkv=2, D=64, P=16,
                           lens_prefill=[5, 16, 31], n_append=20, seed=2)
    k, v = W.gen_pool(wl)
    kn, vn = W.gen_append(wl)
    k2, v2, lens2 = oracle.append_kv(k, v, wl.block_table, wl.lens_prefill, kn, vn)
    np.testing.assert_array_equal(lens2, wl.lens_prefill + 20)
    touched = np.zeros(k.shape[:1] + k.shape[2:3], bool)      # [page, slot]
    for b in range(wl.B):
        L0 = int(wl.lens_prefill[b])
        for name, pool, new, before in (("k", k2, kn, k), ("v", v2, vn, v)):
            logical = np_gather(pool, wl.block_table, b, L0 + 20)
            np.testing.assert_array_equal(logical[:L0], np_gather(before, wl.block_table, b, L0))
            np.testing.assert_array_equal(logical[L0:], new[b])
            got = oracle.gather_kv(pool, wl.block_table, lens2, b)
            np.testing.assert_array_equal(got, logical)
        pos = np.arange(L0, L0 + 20)
        touched[wl.block_table[b, pos // 16], pos % 16] = True
    np.testing.assert_array_equal(k2.transpose(0, 2, 1, 3)[~touched], k.transpose(0, 2, 1, 3)[~touched])
    np.testing.assert_array_equal(v2.transpose(0, 2, 1, 3)[~touched], v.transpose(0, 2, 1, 3)[~touched])


def test_bad_page_index_is_reported():
    wl, q, k, v = small([20])
    bt = wl.block_table.copy()
    bt[0, 1] = wl.num_pages          # outside the pool
    with pytest.raises(RuntimeError, match="page index"):
        oracle.decode_attention(q, k, v, bt, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                scale=wl.scale)


def test_memory_accounting_eq8_eq9():
    """PrefillShare Eqs. 8-9 with no per-model tail: the shared layout holds
    one copy of every request's context, the per-model layout N copies."""
    lens = [1, 16, 17, 1000]
    P = 16
    one = 1 + 1 + 2 + 63
    assert W.pages_required(lens, P, n_models=4, shared=True) == one
    assert W.pages_required(lens, P, n_models=4, shared=False) == 4 * one
