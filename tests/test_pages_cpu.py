"""The page manager (host only) against a plain Python model of its policy.

Policy (PrFaaS hybrid prefix cache pool; ICaRus key design 2): full,
block-aligned blocks of a prompt are reusable prefix-cache pages, matched by
the exact token prefix they end; a partial last block is never reused;
transfer pages are never indexed and are freed on release; an unreferenced
prefix page stays cached until an allocation needs a page, oldest idle page
first; free pages are handed out lowest first, released ones last-in
first-out.  The model below restates that policy with Python containers and
exact token-tuple keys (no hashing); the library must agree with it on every
page id, hit length, reference count and count of pages per state.
"""
import numpy as np
import pytest

from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return N.load()


def make(num_pages, P):
    from cross_model_shared_gb300 import PrefixPages
    return PrefixPages(num_pages, P)


class Model:
    def __init__(self, num_pages, P):
        self.P = P
        self.ref = [0] * num_pages
        self.state = ["free"] * num_pages
        self.free = list(range(num_pages - 1, -1, -1))     # stack: the last item is handed out next
        self.index = {}                                     # token prefix (tuple) -> page
        self.key = {}                                       # page -> its token prefix
        self.idle = []                                      # idle indexed pages, oldest first
        self.lookups = self.hits = 0

    def _take(self):
        if self.free:
            return self.free.pop()
        if self.idle:
            pg = self.idle.pop(0)
            del self.index[self.key.pop(pg)]
            return pg
        return None

    def _drop(self, pg):
        self.ref[pg] -= 1
        if self.ref[pg] == 0:
            if self.state[pg] == "prefix":
                self.idle.append(pg)
            else:
                self.state[pg] = "free"
                self.free.append(pg)

    def acquire(self, tokens):
        P = self.P
        nb = (len(tokens) + P - 1) // P
        pages = []
        while len(pages) < len(tokens) // P and tuple(tokens[:(len(pages) + 1) * P]) in self.index:
            pages.append(self.index[tuple(tokens[:(len(pages) + 1) * P])])
        hit = len(pages)
        self.lookups += len(tokens) // P
        self.hits += hit
        for pg in pages:
            if pg in self.idle:
                self.idle.remove(pg)
            self.ref[pg] += 1
        for _ in range(hit, nb):
            pg = self._take()
            if pg is None:
                for q in reversed(pages):
                    self._drop(q)
                raise MemoryError
            self.state[pg] = "private"
            self.ref[pg] = 1
            pages.append(pg)
        return pages, hit * P

    def publish(self, tokens, pages):
        for i in range(len(tokens) // self.P):
            key = tuple(tokens[:(i + 1) * self.P])
            pg = pages[i]
            if self.state[pg] == "private" and key not in self.index:
                self.index[key] = pg
                self.key[pg] = key
                self.state[pg] = "prefix"

    def release(self, pages):
        for pg in pages:
            self._drop(pg)

    def alloc_transfer(self, n):
        out = []
        for _ in range(n):
            pg = self._take()
            if pg is None:
                for q in reversed(out):
                    self._drop(q)
                raise MemoryError
            self.state[pg] = "transfer"
            self.ref[pg] = 1
            out.append(pg)
        return out

    def stats(self):
        return {"num_pages": len(self.ref), "free_pages": len(self.free), "cached_idle_pages": len(self.idle),
                "referenced_pages": sum(r > 0 for r in self.ref), "indexed_blocks": len(self.index),
                "transfer_pages": sum(s == "transfer" for s in self.state), "block_lookups": self.lookups,
                "block_hits": self.hits}


def agree(lib_pages, model):
    assert lib_pages.stats() == model.stats()
    for pg in range(len(model.ref)):
        assert lib_pages.refcount(pg) == model.ref[pg], pg


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_agree_with_the_model(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([2, 4, 16]))
    num_pages = int(rng.integers(6, 40))
    lib_pages, model = make(num_pages, P), Model(num_pages, P)
    # prompts grow out of a few shared stems, the agent workflow shape
    stems = [list(rng.integers(0, 5, size=int(rng.integers(0, 4 * P)))) for _ in range(3)]
    live, transfers = [], []
    for _ in range(300):
        op = rng.random()
        if op < 0.5:
            stem = stems[int(rng.integers(0, len(stems)))]
            cut = int(rng.integers(0, len(stem) + 1))
            prompt = [int(x) for x in stem[:cut]] + [int(x) for x in rng.integers(0, 5, size=int(rng.integers(0, 3 * P)))]
            try:
                want = model.acquire(prompt)
            except MemoryError:
                want = None
            if want is None:
                with pytest.raises(N.ShkvError) as e:
                    lib_pages.acquire(prompt)
                assert e.value.status == N.SHKV_ERR_CAPACITY
            else:
                got_pages, got_hit = lib_pages.acquire(prompt)
                assert list(got_pages) == want[0] and got_hit == want[1]
                if rng.random() < 0.7:
                    model.publish(prompt, want[0])
                    lib_pages.publish(prompt, got_pages)
                live.append(want[0])
        elif op < 0.8 and live:
            pages = live.pop(int(rng.integers(0, len(live))))
            model.release(pages)
            lib_pages.release(pages)
        elif op < 0.9:
            n = int(rng.integers(0, 4))
            try:
                want = model.alloc_transfer(n)
            except MemoryError:
                want = None
            if want is None:
                with pytest.raises(N.ShkvError):
                    lib_pages.alloc_transfer(n)
            else:
                assert list(lib_pages.alloc_transfer(n)) == want
                transfers.append(want)
        elif transfers:
            pages = transfers.pop(0)
            model.release(pages)
            lib_pages.release(pages)
        agree(lib_pages, model)


def test_only_full_blocks_are_reused():
    m = make(16, 4)
    prompt = list(range(10))                       # 2 full blocks + 2 tokens
    pages, hit = m.acquire(prompt)
    assert hit == 0 and len(pages) == 3
    m.publish(prompt, pages)
    again, hit = m.acquire(prompt)
    assert hit == 8 and list(again[:2]) == list(pages[:2]) and again[2] != pages[2]
    assert m.refcount(int(pages[0])) == 2 and m.refcount(int(pages[2])) == 1


def test_a_hit_needs_the_same_prefix_not_just_the_same_block():
    m = make(16, 4)
    a = [1, 2, 3, 4, 5, 6, 7, 8]
    pa, _ = m.acquire(a)
    m.publish(a, pa)
    b = [9, 9, 9, 9, 5, 6, 7, 8]                  # second block equal, first differs
    _, hit = m.acquire(b)
    assert hit == 0


def test_transfer_pages_are_never_indexed_and_are_freed():
    m = make(8, 4)
    tp = m.alloc_transfer(3)
    with pytest.raises(N.ShkvError) as e:
        m.publish([0, 1, 2, 3], tp[:1])
    assert e.value.status == N.SHKV_ERR_INVALID_ARG
    assert m.stats()["transfer_pages"] == 3
    m.release(tp)
    s = m.stats()
    assert s["transfer_pages"] == 0 and s["free_pages"] == 8 and s["indexed_blocks"] == 0


def test_idle_cached_pages_are_evicted_oldest_first_only_when_needed():
    m = make(4, 2)
    a, b = [1, 1], [2, 2]
    pa, _ = m.acquire(a)
    m.publish(a, pa)
    pb, _ = m.acquire(b)
    m.publish(b, pb)
    m.release(pa)
    m.release(pb)
    assert m.stats()["cached_idle_pages"] == 2
    x, _ = m.acquire([7, 7, 7, 7])                 # two free pages are left: no eviction
    assert m.stats()["cached_idle_pages"] == 2
    y, _ = m.acquire([8, 8])                       # evicts a's page, the oldest idle one
    assert list(y) == list(pa)
    pb2, hit_b = m.acquire(b)                      # b is still cached
    assert hit_b == 2 and list(pb2) == list(pb)
    m.release(pb2)
    pa2, hit_a = m.acquire(a)                      # a was evicted: a miss, on b's idle page
    assert hit_a == 0 and list(pa2) == list(pb)


def test_capacity_error_keeps_everything_as_it_was():
    m = make(3, 2)
    p, _ = m.acquire([1, 2, 3, 4])
    m.publish([1, 2, 3, 4], p)
    before = m.stats()
    with pytest.raises(N.ShkvError) as e:
        m.acquire([1, 2, 3, 4, 5, 6, 7, 8])       # 2 hits + 2 new pages, 1 free
    assert e.value.status == N.SHKV_ERR_CAPACITY
    after = m.stats()
    before.pop("block_lookups"), after.pop("block_lookups")
    before.pop("block_hits"), after.pop("block_hits")
    assert after == before
    assert [m.refcount(i) for i in range(3)] == [1, 1, 0]
