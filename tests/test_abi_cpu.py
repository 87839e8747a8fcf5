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
    assert lib.shkv_selftest_bounded_wait(None, None) == N.SHKV_ERR_INVALID_ARG


def plan_costs(consumer, P, rows):
    """The cost model the header documents for shkv_plan_decode, in tokens:
    (stage, per piece, extra for an opening split piece, extra for a closing
    split piece)."""
    if consumer == N.SHKV_CONSUMER_TCGEN05 and rows <= 16:
        return 128, 7 * rows, 4 * rows, 23 * rows
    if consumer == N.SHKV_CONSUMER_TCGEN05:
        return 128, 12 * rows, 5 * rows, 28 * rows
    return min(P, 32), 16 * P, 0, 0


def range_costs(begin, lens, P, H, costs):
    """Brute force: each range's cost, piece by piece (stage grid from the
    piece's first page)."""
    stage, seg, first, last = costs
    units, off = [], 0
    for l in lens:
        pg = -(-l // P)
        for _ in range(H):
            units.append((off, off + pg))
            off += pg
    out = []
    for c in range(len(begin) - 1):
        a, b = int(begin[c]), int(begin[c + 1])
        t = 0
        for u0, u1 in units:
            lo, hi = max(a, u0), min(b, u1)
            if lo < hi:
                t += -(-(hi - lo) * P // stage) * stage + seg + (first if lo > u0 else 0) + (last if hi < u1 else 0)
        out.append(t)
    return np.array(out), units


@pytest.mark.parametrize("consumer", [N.SHKV_CONSUMER_MMA_SYNC, N.SHKV_CONSUMER_TCGEN05])
@pytest.mark.parametrize("lens,P,H,NM,HQ,C", [
    ([256], 16, 2, 2, 16, 152),                        # tiny
    ([1, 2, 3, 4000, 17], 16, 8, 4, 32, 152),
    ([131584] * 4, 16, 8, 8, 16, 152),                 # long context: every unit split
    (list(range(1, 300)), 32, 8, 8, 40, 152),
    ([5], 16, 1, 1, 16, 152),                          # fewer chunks than CTAs
    ([512] * 40 + [32768] * 3, 16, 8, 4, 32, 152),     # many short requests next to long ones
    ([1 + (37 * i) % 96 for i in range(1024)], 16, 8, 2, 32, 152),   # the largest batch, ragged
    ([1] * 1024, 32, 2, 1, 32, 152),                   # the largest batch, one token each
    ([70000, 3, 9000, 1, 65536], 64, 4, 2, 16, 7),     # pages larger than a stage, few CTAs
])
def test_plan_covers_every_chunk_with_balanced_cost(lib, consumer, lens, P, H, NM, HQ, C):
    begin, nc, ns = N.shkv_plan_decode(lens, P, H, NM, HQ, consumer, C)
    pages = [(l + P - 1) // P for l in lens]
    W = H * sum(pages)
    assert begin[0] == 0 and begin[-1] == W and len(begin) == nc + 1
    assert (np.diff(begin) >= 1).all()                          # every CTA owns work
    c_max = min(C, max(1, -(-W // 8)))
    assert 1 <= nc <= c_max
    costs = plan_costs(consumer, P, NM * HQ // H)
    cost, units = range_costs(begin, lens, P, H, costs)
    cuts = begin.tolist()
    n_split = sum(1 for u0, u1 in units if any(u0 < c < u1 for c in cuts[1:-1]))
    assert ns == n_split and ns <= nc - 1
    # the bisection's bound: within a stage step and one split's fixed costs
    # of the mean over c_max ranges, to its tolerance
    stage, seg, first, last = costs
    step = -(-max(1, stage // P) * P // stage) * stage
    whole = H * sum(seg + -(-pg * P // stage) * stage for pg in pages)
    tol = max(16, whole // c_max // 2048)
    assert cost.max() <= -(-whole // c_max) + seg + first + last + step + tol, (cost.max(), whole / c_max)


def test_plan_cuts_on_the_stage_grid_of_each_piece(lib):
    """tcgen05 plan: a cut inside a (request, head) leaves the piece before it
    a whole number of 128-token stages, counted from the piece's first page."""
    lens = [131584] * 4 + [5000, 77, 3000]
    P, H = 16, 8
    begin, nc, ns = N.shkv_plan_decode(lens, P, H, 8, 16, N.SHKV_CONSUMER_TCGEN05, 152)
    assert ns >= 32                                  # every long unit is cut, many times over
    _, units = range_costs(begin, lens, P, H, plan_costs(N.SHKV_CONSUMER_TCGEN05, P, 16))
    cuts = begin.tolist()
    for u0, u1 in units:
        inner = [c for c in cuts[1:-1] if u0 < c < u1]
        for a, b in zip([u0] + inner, inner):
            assert (b - a) % (128 // P) == 0


def test_plan_is_repeatable_and_follows_its_inputs(lib):
    """Equal inputs give equal plans (the host keeps each thread's last plan
    and reuses it only for identical inputs); another consumer or one more
    page re-plans."""
    lens = [int(x) for x in np.random.default_rng(5).integers(1, 9000, 64)]
    T, M = N.SHKV_CONSUMER_TCGEN05, N.SHKV_CONSUMER_MMA_SYNC
    a = N.shkv_plan_decode(lens, 16, 8, 4, 32, T, 152)
    b = N.shkv_plan_decode(lens, 16, 8, 4, 32, T, 152)
    assert np.array_equal(a[0], b[0]) and a[1:] == b[1:]
    m = N.shkv_plan_decode(lens, 16, 8, 4, 32, M, 152)
    assert not np.array_equal(a[0], m[0])
    lens2 = list(lens)
    lens2[7] = (lens2[7] + 15) // 16 * 16 + 1        # one more page for one request
    c = N.shkv_plan_decode(lens2, 16, 8, 4, 32, T, 152)
    assert c[0][-1] == a[0][-1] + 8
    d = N.shkv_plan_decode(lens, 16, 8, 4, 32, T, 152)
    assert np.array_equal(a[0], d[0]) and a[1:] == d[1:]


def test_plan_rejects_bad_arguments(lib):
    T = N.SHKV_CONSUMER_TCGEN05
    for args, status in [
        (([3, 0, 5], 16, 2, 1, 2, T, 152), N.SHKV_ERR_INVALID_ARG),                 # an empty request
        (([1] * (N.SHKV_MAX_BATCH + 1), 16, 2, 1, 2, T, 152), N.SHKV_ERR_INVALID_ARG),
        (([5], 16, 2, 1, 2, 7, 152), N.SHKV_ERR_INVALID_ARG),                      # unknown consumer
        (([5], 16, 2, 1, 2, N.SHKV_CONSUMER_AUTO, 152), N.SHKV_ERR_INVALID_ARG),   # AUTO needs a pool
        (([5], 16, 2, 0, 2, T, 152), N.SHKV_ERR_INVALID_ARG),                      # no decoders
        (([5], 16, 2, 1, 2, T, 0), N.SHKV_ERR_INVALID_ARG),                        # no CTAs
        (([5], 256, 2, 1, 2, T, 152), N.SHKV_ERR_INVALID_ARG),                     # page_size above 255
        (([5], 16, 2, 1, 3, T, 152), N.SHKV_ERR_UNSUPPORTED),                      # hq % hkv
        (([5], 16, 2, 9, 16, T, 152), N.SHKV_ERR_UNSUPPORTED),                     # 72 rows per KV head
    ]:
        with pytest.raises(N.ShkvError) as e:
            N.shkv_plan_decode(*args)
        assert e.value.status == status, args


def test_header_constants_match_binding():
    text = open(HEADER).read()
    for name in ("SHKV_MAX_BATCH", "SHKV_NOALLOC_SCRATCH_BYTES", "SHKV_COUNT_REGION_BYTES"):
        m = re.search(rf"#define {name} \(?(\d+)u?(?: << (\d+))?\)?", text)
        assert m, name
        value = int(m.group(1)) << int(m.group(2) or 0)
        assert getattr(N, name) == value, name
