"""Pins for the oracle's partial-prefill attention (PrefillShare Sec. 3.3:
on a prefix-cache hit the shared prefill module runs only on the new tokens;
each new token attends the cached prefix and the new tokens up to itself).

Checked against the decode oracle where the two coincide, a scipy brute
force over numpy gathers, the causal structure, and closed forms.
"""
import numpy as np
import pytest
import scipy.special

import oracle
from cross_model_shared_gb300 import workloads as W


def widen(bits):
    return W.f32_from_bf16_bits(bits).astype(np.float64)


def setup(lens_total, n_new, Hq=4, Hkv=2, D=64, P=16, seed=31):
    wl = W.custom_workload("prefill", B=len(lens_total), N=1, Hq=Hq, Hkv=Hkv, D=D, P=P, lens_prefill=lens_total,
                           seed=seed)
    rng = np.random.default_rng(seed + 1)
    q = W.bf16_bits_from_f32(rng.standard_normal((wl.B, n_new, Hq, D)).astype(np.float32))
    k, v = W.gen_pool(wl)
    return wl, q, k, v


def run(wl, q, k, v):
    return oracle.prefill_attention(q, k, v, wl.block_table, wl.lens_final, scale=wl.scale)


def test_one_new_token_is_the_decode_oracle():
    wl, q, k, v = setup([5, 40, 17], 1)
    out, lse = run(wl, q, k, v)
    ref, lref = oracle.decode_attention(q[:, 0], k, v, wl.block_table, wl.lens_final, n_models=1, hq=wl.Hq,
                                        scale=wl.scale)
    np.testing.assert_array_equal(out[:, 0], ref)
    np.testing.assert_array_equal(lse[:, 0], lref)


def test_last_new_token_attends_the_whole_cache():
    wl, q, k, v = setup([37, 64, 20], 9)
    out, lse = run(wl, q, k, v)
    ref, lref = oracle.decode_attention(q[:, -1], k, v, wl.block_table, wl.lens_final, n_models=1, hq=wl.Hq,
                                        scale=wl.scale)
    np.testing.assert_array_equal(out[:, -1], ref)
    np.testing.assert_array_equal(lse[:, -1], lref)


def test_brute_force_causal_softmax():
    wl, q, k, v = setup([23, 50, 7], 7, Hq=6, Hkv=2)
    out, lse = run(wl, q, k, v)
    T = q.shape[1]
    for b, L in enumerate(wl.lens_final):
        t = np.arange(L)
        kb = widen(k[wl.block_table[b, t // wl.P], :, t % wl.P, :])     # [L, Hkv, D]
        vb = widen(v[wl.block_table[b, t // wl.P], :, t % wl.P, :])
        for i in range(T):
            pos = L - T + i
            for h in range(wl.Hq):
                g = h // (wl.Hq // wl.Hkv)
                s = wl.scale * kb[:pos + 1, g] @ widen(q[b, i, h])
                np.testing.assert_allclose(out[b, i, h], scipy.special.softmax(s) @ vb[:pos + 1, g], rtol=0,
                                           atol=1e-12)
                assert lse[b, i, h] == pytest.approx(scipy.special.logsumexp(s), abs=1e-12)


def test_a_new_token_never_sees_later_tokens():
    """Changing new token j's K and V changes exactly the queries at
    positions >= j."""
    wl, q, k, v = setup([40], 6)
    out, _ = run(wl, q, k, v)
    L, T = int(wl.lens_final[0]), 6
    j = 3
    pos = L - T + j
    page, slot = wl.block_table[0, pos // wl.P], pos % wl.P
    k2, v2 = k.copy(), v.copy()
    k2[page, :, slot] ^= 0x0101
    v2[page, :, slot] ^= 0x0101
    out2, _ = run(wl, q, k2, v2)
    np.testing.assert_array_equal(out2[0, :j], out[0, :j])
    assert (np.abs(out2[0, j:] - out[0, j:]).max(axis=(1, 2)) > 0).all()


def test_all_new_request_first_token_returns_its_value():
    """No cached prefix (L = n_new): the first new token attends only itself."""
    wl, q, k, v = setup([5], 5, Hq=2, Hkv=1)
    out, lse = run(wl, q, k, v)
    page = wl.block_table[0, 0]
    for h in range(2):
        np.testing.assert_array_equal(out[0, 0, h], widen(v[page, 0, 0]))
        assert lse[0, 0, h] == pytest.approx(wl.scale * widen(q[0, 0, h]) @ widen(k[page, 0, 0]), abs=1e-13)
