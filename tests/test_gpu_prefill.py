"""Causal partial-prefill attention on the tensor cores against the fp64
oracle (PrefillShare Sec. 3.3: on a prefix-cache hit the shared prefill
module runs only on the new tokens; new token i attends the cached prefix
and the new tokens up to itself)."""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, make_pool, torch_to_bits

pytestmark = pytest.mark.gpu

SHAPES = {
    "g4_p16": dict(Hq=32, Hkv=8, P=16),     # Llama-3.1-8B heads: 32 new tokens per tile
    "g5_p32": dict(Hq=40, Hkv=8, P=32),     # Qwen3-14B heads: 25 per tile, 3 padding rows
    "g1_p32": dict(Hq=8, Hkv=8, P=32),      # 128 per tile
    "g8_p16": dict(Hq=16, Hkv=2, P=16),     # 16 per tile
    "g16_p32": dict(Hq=32, Hkv=2, P=32),    # 8 per tile
}


def setup(shape, prefix, n_new, seed=41):
    sh = SHAPES[shape]
    lens = [p + n_new for p in prefix]
    wl = W.custom_workload(shape, B=len(lens), N=1, Hq=sh["Hq"], Hkv=sh["Hkv"], D=128, P=sh["P"],
                           lens_prefill=lens, seed=seed)
    rng = np.random.default_rng(seed + 3)
    q = W.bf16_bits_from_f32(rng.standard_normal((wl.B, n_new, wl.Hq, 128)).astype(np.float32))
    k, v = W.gen_pool(wl)
    return wl, q, k, v, make_pool(wl, k, v)


def check(wl, q, k, v, pool, what):
    out, lse = pool.prefill_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    ref, lref = oracle.prefill_attention(q, k, v, wl.block_table, wl.lens_final, scale=wl.scale)
    compare(out, ref, lse, lref, what=what)
    return out, lse


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_prefill_matches_oracle(shape):
    wl, q, k, v, pool = setup(shape, [0, 1, 127, 128, 129, 700], 41)
    check(wl, q, k, v, pool, f"prefill {shape}")


@pytest.mark.parametrize("n_new", [1, 7, 64, 200, 300])
def test_prefill_new_token_counts(n_new):
    wl, q, k, v, pool = setup("g5_p32", [5, 1000, 0], n_new, seed=n_new)
    check(wl, q, k, v, pool, f"n_new {n_new}")


def test_append_then_prefill_last_token_matches_decode():
    """The normal flow: append the new tokens' K/V, then run the prefill;
    its last token attends the whole cache, like a decode of that query."""
    n_new = 50
    prefix = [300, 17]
    sh = SHAPES["g4_p16"]
    wl = W.custom_workload("flow", B=2, N=1, Hq=sh["Hq"], Hkv=sh["Hkv"], D=128, P=sh["P"], lens_prefill=prefix,
                           n_append=n_new, seed=8)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v, lens=wl.lens_prefill)
    kn, vn = W.gen_append(wl)
    pool.append_kv(bits_to_torch(kn), bits_to_torch(vn))
    rng = np.random.default_rng(5)
    q = W.bf16_bits_from_f32(rng.standard_normal((2, n_new, wl.Hq, 128)).astype(np.float32))
    out, lse = pool.prefill_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    k2, v2 = torch_to_bits(pool.k_pages), torch_to_bits(pool.v_pages)
    ref, lref = oracle.prefill_attention(q, k2, v2, wl.block_table, wl.lens_final, scale=wl.scale)
    compare(out, ref, lse, lref, what="append + prefill")
    dec, dlse = pool.decode_attention(bits_to_torch(np.ascontiguousarray(q[:, -1])), 1, scale=wl.scale,
                                      return_lse=True)
    compare(out[:, -1], dec.double().cpu().numpy(), what="last token vs decode")


def test_earlier_tokens_are_unaffected_by_later_ones():
    """Changing new token j's K/V leaves every earlier new token's output
    bit-identical on the GPU (the causal mask removes it exactly)."""
    wl, q, k, v, pool = setup("g5_p32", [600], 60)
    out1 = pool.prefill_attention(bits_to_torch(q), scale=wl.scale).clone()
    j = 37
    pos = int(wl.lens_final[0]) - 60 + j
    page, slot = wl.block_table[0, pos // wl.P], pos % wl.P
    pool.k_pages[page, :, slot] = pool.k_pages[page, :, slot] * 3
    pool.v_pages[page, :, slot] = pool.v_pages[page, :, slot] * -2
    out2 = pool.prefill_attention(bits_to_torch(q), scale=wl.scale)
    assert torch.equal(out1[0, :j], out2[0, :j])
    assert not torch.equal(out1[0, j:], out2[0, j:])


def test_long_prefix_qwen14b_shape_sampled():
    """27K-token cached prefixes, 512 new tokens, Qwen3-14B heads; checked on
    sampled rows against the oracle."""
    n_new = 512
    prefix = [27648, 9000]
    wl, q, k, v, pool = setup("g5_p32", prefix, n_new, seed=77)
    out, lse = pool.prefill_attention(bits_to_torch(q), scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    rows = [0, 1, 255, 511]
    # rows at positions prefix + i: attend keys 0 .. prefix + i; the oracle on
    # a one-token prefill over truncated lengths reproduces each row
    for i in rows:
        lens_i = (np.asarray(prefix) + i + 1).astype(np.int32)
        r1, l1 = oracle.prefill_attention(np.ascontiguousarray(q[:, i:i + 1]), k, v, wl.block_table, lens_i,
                                          scale=wl.scale)
        compare(out[:, i:i + 1], r1, lse[:, i:i + 1], l1, what=f"long prefix row {i}")


def test_out_of_range_page_sets_flag():
    wl, q, k, v, pool = setup("g4_p16", [200, 200], 30)
    pool.block_table[1, 2] = wl.num_pages + 9
    out = pool.prefill_attention(bits_to_torch(q), scale=wl.scale)
    assert pool.check_errors() & N.SHKV_ERRF_PAGE_OOB
    assert bool(torch.isfinite(out.float()).all())
