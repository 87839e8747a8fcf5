"""Prefix-cache pages shared across requests and decoder models, end to end.

ICaRus key design 2: every task model's encoder is the frozen base, so a
prompt's KV cache is a function of the tokens alone and a prefix cached for
one agent is reusable by every later agent; PrFaaS: only block-aligned, full
blocks are reused.  Here K/V of a token are a fixed function of (token id,
position) - the stand-in for the frozen base encoder - so a prefix hit must
give exactly the cache a fresh prefill would have written.
"""
import numpy as np
import pytest
import torch

import oracle
from cross_model_shared_gb300 import PrefixPages
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, torch_to_bits
from cross_model_shared_gb300 import SharedKVPool

pytestmark = pytest.mark.gpu

N_MODELS, HQ, HKV, D, P = 4, 8, 2, 128, 16


def base_kv(tokens, start, rng_table):
    """bf16 K/V [T, Hkv, D] of tokens at positions start.. (deterministic)."""
    t = np.asarray(tokens)
    pos = np.arange(start, start + len(t))
    idx = (t * 7919 + pos) % rng_table.shape[0]
    return rng_table[idx]


def test_cross_agent_prefix_hit_reuses_pages_and_matches_the_oracle():
    rng = np.random.default_rng(21)
    table_k = W.bf16_bits_from_f32(rng.standard_normal((4096, HKV, D)).astype(np.float32))
    table_v = W.bf16_bits_from_f32(rng.standard_normal((4096, HKV, D)).astype(np.float32))
    num_pages = 64
    pages = PrefixPages(num_pages, P)
    pool = SharedKVPool(num_pages, P, HKV, D, max_batch=3, max_pages_per_seq=16, initial_seq_lens=[0, 0, 0])
    vocab = rng.integers(0, 1000, size=400)
    prompt_a = [int(x) for x in vocab[:75]]                 # planner: 4 full blocks + 11 tokens
    prompt_b = prompt_a[:70] + [int(x) for x in vocab[200:260]]   # executor: shares 4 full blocks

    def admit(b, prompt):
        pg, cached = pages.acquire(prompt)
        pool.block_table[b, :len(pg)] = torch.from_numpy(pg).cuda()
        lens = pool.host_seq_lens(3)
        lens[b] = cached
        pool.set_seq_lens(lens)
        new = prompt[cached:]                               # only the uncached tokens are prefilled
        pool_single_append(pool, b, base_kv(new, cached, table_k), base_kv(new, cached, table_v))
        pages.publish(prompt, pg)
        return pg, cached

    pa, ca = admit(0, prompt_a)
    pb, cb = admit(1, prompt_b)
    assert ca == 0 and cb == 64
    assert list(pb[:4]) == list(pa[:4]) and not set(pb[4:]) & set(pa)
    assert all(pages.refcount(int(x)) == 2 for x in pa[:4])
    assert pool.check_errors() == 0

    # decode both requests: N decoders stacked over each request's cache
    q = W.bf16_bits_from_f32(rng.standard_normal((2, N_MODELS * HQ, D)).astype(np.float32))
    out, lse = pool.decode_attention(bits_to_torch(q), N_MODELS, return_lse=True)
    k_all, v_all = torch_to_bits(pool.k_pages), torch_to_bits(pool.v_pages)
    bt = pool.block_table[:2].cpu().numpy()
    lens = pool.host_seq_lens(2)
    assert list(lens) == [len(prompt_a), len(prompt_b)]
    ref, lref = oracle.decode_attention(q, k_all, v_all, bt, lens, n_models=N_MODELS, hq=HQ, scale=D ** -0.5)
    compare(out, ref, lse, lref, what="prefix pages")

    # the shared pages hold exactly what a fresh prefill of prompt_b writes
    t = np.arange(len(prompt_b))
    cache_b = k_all[bt[1, t // P], :, t % P, :]
    np.testing.assert_array_equal(cache_b, base_kv(prompt_b, 0, table_k))

    # and sharing changes nothing: private copies of every page, same plan
    priv = SharedKVPool(num_pages, P, HKV, D, max_batch=2, max_pages_per_seq=16, initial_seq_lens=list(lens))
    k2, v2 = np.zeros_like(k_all), np.zeros_like(v_all)
    nxt = 0
    bt2 = np.full((2, 16), -1, np.int32)
    for b in range(2):
        for i in range((int(lens[b]) + P - 1) // P):
            k2[nxt], v2[nxt] = k_all[bt[b, i]], v_all[bt[b, i]]
            bt2[b, i] = nxt
            nxt += 1
    priv.k_pages.copy_(bits_to_torch(k2))
    priv.v_pages.copy_(bits_to_torch(v2))
    priv.block_table.copy_(torch.from_numpy(bt2).cuda())
    out2, lse2 = priv.decode_attention(bits_to_torch(q), N_MODELS, return_lse=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)

    # releasing the planner keeps the shared blocks alive for the executor
    pages.release(pa)
    assert all(pages.refcount(int(x)) == 1 for x in pa[:4])
    assert pages.refcount(int(pa[4])) == 0


def pool_single_append(pool, b, k_new, v_new):
    """Append T tokens to request b only: a one-request view of the same
    pages (shkv_append_kv appends to requests 0..batch-1)."""
    T = k_new.shape[0]
    if T == 0:
        return
    view = SharedKVPool(pool.num_pages, pool.page_size, pool.num_kv_heads, pool.head_dim, max_batch=1,
                        max_pages_per_seq=pool.max_pages_per_seq, k_pages=pool.k_pages, v_pages=pool.v_pages,
                        initial_seq_lens=[int(pool.host_seq_lens(b + 1)[b])])
    view.block_table[0].copy_(pool.block_table[b])
    torch.cuda.synchronize()
    view.append_kv(bits_to_torch(k_new[None]), bits_to_torch(v_new[None]))
    assert view.check_errors() == 0
    lens = pool.host_seq_lens(pool.max_batch)
    lens[b] += T
    pool.set_seq_lens(lens)
