"""CPU-side checks of the C ABI: the library loads, exports every symbol the
header declares, and its host-only entry points (status strings, the split
plan) behave.  No compute call is made without a GPU."""
import os
import re

import numpy as np
import pytest

from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "shkv.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(shkv_\w+)\s*\(", text, re.M)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(N.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    syms = os.popen(f"nm -D --defined-only {N.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", syms), f"{name} not exported"


def test_status_strings(lib):
    for st in range(6):
        assert N.status_string(st)
    assert N.status_string(N.SHKV_OK) == "ok"


def test_null_arguments_are_rejected_without_a_device(lib):
    assert lib.shkv_pool_create(None, None) == N.SHKV_ERR_INVALID_ARG
    assert lib.shkv_pool_destroy(None) == N.SHKV_ERR_INVALID_ARG
    assert lib.shkv_decode_attention(None, 1, 1, 1, None, 1.0, None, None, None, 0, None) == N.SHKV_ERR_INVALID_ARG
    assert lib.shkv_splitkv_merge(0, 1, 1, 4, None, None, None, None, None) == N.SHKV_ERR_INVALID_ARG
    assert lib.shkv_splitkv_merge(1, 1, 1, 6, 16, 16, 16, None, None) == N.SHKV_ERR_INVALID_ARG  # D % 4
    assert lib.shkv_pool_set_decode_consumer(None, 0) == N.SHKV_ERR_INVALID_ARG
    assert lib.shkv_decode_attention_noalloc(None, 1, 1, 1, None, 1.0, None, None, None) == N.SHKV_ERR_INVALID_ARG


SEGMENT_COST = 16  # chunks charged per (request, head) segment by the planner


@pytest.mark.parametrize("lens,P,H,C", [
    ([256], 16, 2, 152),                       # tiny
    ([1, 2, 3, 4000, 17], 16, 8, 152),
    ([131584] * 4, 16, 8, 152),                # long context: every unit split
    (list(range(1, 300)), 32, 8, 152),
    ([5], 16, 1, 152),                         # fewer chunks than CTAs
    ([512] * 40 + [32768] * 3, 16, 8, 152),    # many short requests next to long ones
    ([1 + (37 * i) % 96 for i in range(1024)], 16, 8, 152),   # the largest batch, ragged
    ([1] * 1024, 32, 2, 152),                  # the largest batch, one token each
])
def test_plan_covers_every_chunk_with_balanced_cost(lib, lens, P, H, C):
    begin, nc, ns = N.shkv_plan_decode(lens, P, H, C)
    pages = [(l + P - 1) // P for l in lens]
    W = H * sum(pages)
    assert begin[0] == 0 and begin[-1] == W
    sizes = np.diff(begin)
    assert (sizes >= 1).all()                                   # every CTA owns work
    assert nc <= C and nc == min(C, max(1, -(-W // 8)))
    # brute force: segments per CTA and units straddling a cut
    units = []
    off = 0
    for p_ in pages:
        for _ in range(H):
            units.append((off, off + p_))
            off += p_
    cuts = begin.tolist()
    n_split = sum(1 for u0, u1 in units if any(u0 < c < u1 for c in cuts[1:-1]))
    assert ns == n_split and ns <= nc - 1
    cost = []
    for c in range(nc):
        a, b = cuts[c], cuts[c + 1]
        segs = sum(1 for u0, u1 in units if u0 < b and u1 > a)
        cost.append((b - a) + SEGMENT_COST * segs)
    target = (W + SEGMENT_COST * len(units)) / nc
    assert max(cost) <= target + 3 * SEGMENT_COST + 2, (max(cost), target)


def test_plan_rejects_empty_requests_and_oversized_batches(lib):
    with pytest.raises(N.ShkvError):
        N.shkv_plan_decode([3, 0, 5], 16, 2, 152)
    with pytest.raises(N.ShkvError):
        N.shkv_plan_decode([1] * (N.SHKV_MAX_BATCH + 1), 16, 2, 152)
