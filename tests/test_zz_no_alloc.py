"""shkv_decode_attention_noalloc: decode attention for callers that cannot
call cudaMalloc (code inside a framework that owns all device memory and
offers no allocation hook, or on a latency-critical path where cudaMalloc's
implicit synchronisation is not acceptable).  The entry point runs on the
library's static device scratch instead of a caller workspace.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.  It must pass both alone in a
fresh process and after the rest of the suite (the static scratch keeps the
previous call's contents; each call clears what must start at zero).
"""
import pytest
import torch

import oracle
from cross_model_shared_gb300 import _native as N
from cross_model_shared_gb300 import workloads as W
from tests.gpu_common import bits_to_torch, compare, make_pool

pytestmark = pytest.mark.gpu


def _noalloc(pool, q, n_models, scale):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    N.shkv_decode_attention_noalloc(pool.handle, q.shape[0], n_models, q.shape[1] // n_models, q.data_ptr(),
                                    scale, out.data_ptr(), lse.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    return out, lse


SHAPES = [
    (dict(N=2, Hq=32, Hkv=8, D=128, P=16), [40000, 700, 3000, 64]),     # Llama-3.1-8B heads, split units
    (dict(N=8, Hq=40, Hkv=8, D=128, P=32), [5000, 1025, 33]),           # Qwen3-14B heads, R = 40
]


@pytest.mark.parametrize("shape,lens", SHAPES)
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(shape, lens):
    wl = W.custom_workload("noalloc", B=len(lens), lens_prefill=lens, seed=31, **shape)
    q_bits = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    q = bits_to_torch(q_bits)
    ref, ref_lse = pool.decode_attention(q, wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    o64, l64 = oracle.decode_attention(q_bits, k, v, wl.block_table, wl.lens_final, n_models=wl.N, hq=wl.Hq,
                                       scale=wl.scale)
    for call in range(2):
        out, lse = _noalloc(pool, q, wl.N, wl.scale)
        assert pool.check_errors() == 0, f"device error bits on call {call}"
        compare(out, o64, lse, l64, what=f"noalloc call {call} vs oracle")
        # same kernel, same split plan: the same bits as the workspace entry point
        assert torch.equal(out, ref), f"call {call}: output differs from shkv_decode_attention"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from shkv_decode_attention"


def test_noalloc_is_exact_after_a_call_that_set_error_bits():
    """A call over an out-of-range block-table entry (bounds-checked on the
    device: the page is skipped and a flag set) leaves the shared scratch as
    it may; the next call must still give the exact result."""
    shape, lens = SHAPES[0]
    wl = W.custom_workload("noalloc_err", B=len(lens), lens_prefill=lens, seed=37, **shape)
    q_bits = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    q = bits_to_torch(q_bits)
    ref, ref_lse = pool.decode_attention(q, wl.N, scale=wl.scale, return_lse=True)
    assert pool.check_errors() == 0
    saved = int(pool.block_table[0, 5].item())
    pool.block_table[0, 5] = wl.num_pages + 11
    _noalloc(pool, q, wl.N, wl.scale)
    assert pool.check_errors() & N.SHKV_ERRF_PAGE_OOB
    pool.block_table[0, 5] = saved
    for call in range(2):
        out, lse = _noalloc(pool, q, wl.N, wl.scale)
        assert pool.check_errors() == 0, f"device error bits on call {call}"
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse), f"call {call} after the flagged call"


def test_noalloc_rejected_call_enqueues_nothing():
    """Argument errors return before the scratch is touched; the next valid
    call is exact."""
    shape, lens = SHAPES[1]
    wl = W.custom_workload("noalloc_rej", B=len(lens), lens_prefill=lens, seed=41, **shape)
    q_bits = W.gen_q(wl)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    q = bits_to_torch(q_bits)
    ref = pool.decode_attention(q, wl.N, scale=wl.scale)
    with pytest.raises(N.ShkvError) as e:
        _noalloc(pool, q, wl.N, float("nan"))
    assert e.value.status == N.SHKV_ERR_INVALID_ARG
    out, _ = _noalloc(pool, q, wl.N, wl.scale)
    assert pool.check_errors() == 0
    assert torch.equal(out, ref)


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    """64 stacked rows of d=128 need ~10 MB of split scratch on a GB300,
    more than the 8 MiB the library reserves: rejected before any launch."""
    wl = W.custom_workload("big", B=1, N=8, Hq=16, Hkv=2, D=128, P=16, lens_prefill=[100], seed=1)
    k, v = W.gen_pool(wl)
    pool = make_pool(wl, k, v)
    need = N.shkv_decode_workspace_size(pool.handle, wl.B, wl.N, wl.Hq)
    if need <= N.SHKV_NOALLOC_SCRATCH_BYTES:
        pytest.skip(f"this device needs only {need} bytes for R=64")
    with pytest.raises(N.ShkvError) as e:
        _noalloc(pool, bits_to_torch(W.gen_q(wl)), wl.N, wl.scale)
    assert e.value.status == N.SHKV_ERR_UNSUPPORTED
