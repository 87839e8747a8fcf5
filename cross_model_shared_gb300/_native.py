"""ctypes binding of libshkv (include/shkv.h).

Argument marshalling only: every function here forwards to the C entry
point of the same name.  The library is built in-tree by
``cross_model_shared_gb300.build``; if it is missing, loading fails loudly
(there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libshkv.so")

SHKV_OK = 0
SHKV_ERR_INVALID_ARG = 1
SHKV_ERR_CAPACITY = 2
SHKV_ERR_UNSUPPORTED = 3
SHKV_ERR_CUDA = 4
SHKV_ERR_DEVICE = 5

SHKV_ERRF_PAGE_OOB = 0x1
SHKV_ERRF_SEQ_LEN = 0x2
SHKV_ERRF_TIMEOUT = 0x4
SHKV_ERRF_PIPELINE = 0x8

SHKV_MAX_BATCH = 1024

# Every symbol include/shkv.h declares.
EXPORTS = [
    "shkv_pool_create", "shkv_pool_destroy", "shkv_pool_set_seq_lens", "shkv_pool_get_seq_lens",
    "shkv_append_kv", "shkv_decode_workspace_size", "shkv_decode_attention", "shkv_splitkv_merge",
    "shkv_check_errors", "shkv_plan_decode", "shkv_status_string", "shkv_decode_attention_noalloc",
    "shkv_decode_consumer", "shkv_tails_create", "shkv_tails_destroy", "shkv_tails_set_lens",
    "shkv_tails_get_lens", "shkv_tails_append", "shkv_decode_tails_workspace_size",
    "shkv_decode_attention_tails", "shkv_pages_create", "shkv_pages_destroy", "shkv_pages_acquire",
    "shkv_pages_publish", "shkv_pages_release", "shkv_pages_alloc_transfer", "shkv_pages_stats",
    "shkv_pages_refcount", "shkv_prefill_attention", "shkv_pool_set_decode_consumer",
    "shkv_partition_requests", "shkv_selftest_bounded_wait",
]

SHKV_CONSUMER_AUTO = -1
SHKV_CONSUMER_MMA_SYNC = 0
SHKV_CONSUMER_TCGEN05 = 1

SHKV_NOALLOC_SCRATCH_BYTES = 8 << 20
SHKV_COUNT_REGION_BYTES = 1 << 20


class shkv_pool_config(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_batch", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("k_pages", ctypes.c_void_p),
        ("v_pages", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("error_word", ctypes.c_void_p),
        ("initial_seq_lens", ctypes.c_void_p),
    ]


class shkv_tails_config(ctypes.Structure):
    _fields_ = [
        ("max_batch", ctypes.c_int32),
        ("n_models", ctypes.c_int32),
        ("max_tail_pages", ctypes.c_int32),
        ("block_table", ctypes.c_void_p),
        ("tail_lens", ctypes.c_void_p),
        ("initial_tail_lens", ctypes.c_void_p),
    ]


class shkv_pages_info(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32),
        ("free_pages", ctypes.c_int32),
        ("cached_idle_pages", ctypes.c_int32),
        ("referenced_pages", ctypes.c_int32),
        ("indexed_blocks", ctypes.c_int32),
        ("transfer_pages", ctypes.c_int32),
        ("block_lookups", ctypes.c_int64),
        ("block_hits", ctypes.c_int64),
    ]


class ShkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def load() -> ctypes.CDLL:
    """Load libshkv.so (built in-tree).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libshkv.so not found at {LIB_PATH}: build it with "
                          "`python -m cross_model_shared_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, u32p, i32p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p
    sig = {
        "shkv_pool_create": [ctypes.POINTER(shkv_pool_config), ctypes.POINTER(vp)],
        "shkv_pool_destroy": [vp],
        "shkv_pool_set_seq_lens": [vp, i32, i32p, vp],
        "shkv_pool_get_seq_lens": [vp, i32, i32p],
        "shkv_append_kv": [vp, i32, i32, vp, vp, vp],
        "shkv_decode_workspace_size": [vp, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
        "shkv_decode_attention": [vp, i32, i32, i32, vp, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp],
        "shkv_splitkv_merge": [i32, i32, i32, i32, vp, vp, vp, vp, vp],
        "shkv_check_errors": [vp, vp, u32p],
        "shkv_selftest_bounded_wait": [vp, vp],
        "shkv_plan_decode": [i32, i32p, i32, i32, i32, i32, i32, i32, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "shkv_decode_attention_noalloc": [vp, i32, i32, i32, vp, ctypes.c_float, vp, vp, vp],
        "shkv_decode_consumer": [vp, i32, i32, ctypes.POINTER(i32)],
        "shkv_pool_set_decode_consumer": [vp, i32],
        "shkv_partition_requests": [i32, i32p, i32, i32, i32p, vp],
        "shkv_tails_create": [vp, ctypes.POINTER(shkv_tails_config), ctypes.POINTER(vp)],
        "shkv_tails_destroy": [vp],
        "shkv_tails_set_lens": [vp, i32, i32p, vp],
        "shkv_tails_get_lens": [vp, i32, i32p],
        "shkv_tails_append": [vp, i32, i32, vp, vp, vp],
        "shkv_decode_tails_workspace_size": [vp, vp, i32, i32, ctypes.POINTER(ctypes.c_size_t)],
        "shkv_decode_attention_tails": [vp, vp, i32, i32, vp, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp],
        "shkv_pages_create": [i32, i32, ctypes.POINTER(vp)],
        "shkv_pages_destroy": [vp],
        "shkv_pages_acquire": [vp, i32p, i32, i32p, i32, ctypes.POINTER(i32)],
        "shkv_pages_publish": [vp, i32p, i32, i32p],
        "shkv_pages_release": [vp, i32p, i32],
        "shkv_pages_alloc_transfer": [vp, i32, i32p],
        "shkv_pages_stats": [vp, ctypes.POINTER(shkv_pages_info)],
        "shkv_pages_refcount": [vp, i32, ctypes.POINTER(i32)],
        "shkv_prefill_attention": [vp, i32, i32, i32, vp, ctypes.c_float, vp, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.shkv_status_string.argtypes = [ctypes.c_int]
    lib.shkv_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().shkv_status_string(int(status)).decode()


def _check(status: int, what: str) -> int:
    if status != SHKV_OK:
        raise ShkvError(status, what)
    return status


# --- thin wrappers, one per C entry point (pointers are ints) -------------
def shkv_pool_create(cfg: shkv_pool_config) -> int:
    h = ctypes.c_void_p()
    _check(load().shkv_pool_create(ctypes.byref(cfg), ctypes.byref(h)), "shkv_pool_create")
    return h.value


def shkv_pool_destroy(pool: int) -> None:
    _check(load().shkv_pool_destroy(pool), "shkv_pool_destroy")


def shkv_pool_set_seq_lens(pool: int, batch: int, lens_ptr: int, stream: int) -> None:
    _check(load().shkv_pool_set_seq_lens(pool, batch, lens_ptr, stream), "shkv_pool_set_seq_lens")


def shkv_pool_get_seq_lens(pool: int, batch: int, lens_ptr: int) -> None:
    _check(load().shkv_pool_get_seq_lens(pool, batch, lens_ptr), "shkv_pool_get_seq_lens")


def shkv_append_kv(pool: int, batch: int, n_new: int, k_new: int, v_new: int, stream: int) -> None:
    _check(load().shkv_append_kv(pool, batch, n_new, k_new, v_new, stream), "shkv_append_kv")


def shkv_decode_workspace_size(pool: int, batch: int, n_models: int, hq: int) -> int:
    n = ctypes.c_size_t()
    _check(load().shkv_decode_workspace_size(pool, batch, n_models, hq, ctypes.byref(n)),
           "shkv_decode_workspace_size")
    return n.value


def shkv_decode_attention(pool: int, batch: int, n_models: int, hq: int, q: int, scale: float, out: int,
                          lse_out: int, workspace: int, workspace_bytes: int, stream: int) -> None:
    _check(load().shkv_decode_attention(pool, batch, n_models, hq, q, scale, out, lse_out, workspace,
                                        workspace_bytes, stream), "shkv_decode_attention")


def shkv_splitkv_merge(n_splits: int, batch: int, rows: int, head_dim: int, o_part: int, lse_part: int,
                       out: int, lse_out: int, stream: int) -> None:
    _check(load().shkv_splitkv_merge(n_splits, batch, rows, head_dim, o_part, lse_part, out, lse_out, stream),
           "shkv_splitkv_merge")


def shkv_check_errors(pool: int, stream: int) -> int:
    """Returns the device error bits (0 if none); raises only on CUDA errors."""
    flags = ctypes.c_uint32()
    st = load().shkv_check_errors(pool, stream, ctypes.byref(flags))
    if st not in (SHKV_OK, SHKV_ERR_DEVICE):
        raise ShkvError(st, "shkv_check_errors")
    return flags.value


def shkv_selftest_bounded_wait(pool: int, stream: int) -> None:
    _check(load().shkv_selftest_bounded_wait(pool, stream), "shkv_selftest_bounded_wait")


def shkv_plan_decode(lens, page_size: int, num_kv_heads: int, n_models: int, hq_per_model: int, consumer: int,
                     max_ctas: int):
    """Host-only split plan for `consumer` (SHKV_CONSUMER_MMA_SYNC or
    SHKV_CONSUMER_TCGEN05): (cta_begin list, num_ctas, num_splits)."""
    import numpy as np
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    begin = np.zeros(max_ctas + 1, dtype=np.int64)
    nc, ns = ctypes.c_int32(), ctypes.c_int32()
    _check(load().shkv_plan_decode(len(lens), lens.ctypes.data, page_size, num_kv_heads, n_models, hq_per_model,
                                   consumer, max_ctas, begin.ctypes.data, ctypes.byref(nc), ctypes.byref(ns)),
           "shkv_plan_decode")
    return begin[: nc.value + 1].copy(), nc.value, ns.value


def shkv_decode_attention_noalloc(pool: int, batch: int, n_models: int, hq: int, q: int, scale: float, out: int,
                                  lse_out: int, stream: int) -> None:
    """Decode attention on the library's static device scratch (no workspace
    argument, no allocation)."""
    _check(load().shkv_decode_attention_noalloc(pool, batch, n_models, hq, q, scale, out, lse_out, stream),
           "shkv_decode_attention_noalloc")


def shkv_partition_requests(lens, page_size: int, world_size: int):
    """Host-only division of a batch among replicas: (owner int32 [batch],
    pages per replica int64 [world_size])."""
    import numpy as np
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    owner = np.zeros(len(lens), dtype=np.int32)
    rank_pages = np.zeros(world_size, dtype=np.int64)
    _check(load().shkv_partition_requests(len(lens), lens.ctypes.data, page_size, world_size, owner.ctypes.data,
                                          rank_pages.ctypes.data), "shkv_partition_requests")
    return owner, rank_pages


def shkv_pool_set_decode_consumer(pool: int, consumer: int) -> None:
    _check(load().shkv_pool_set_decode_consumer(pool, consumer), "shkv_pool_set_decode_consumer")


def shkv_decode_consumer(pool: int, n_models: int, hq: int) -> int:
    """SHKV_CONSUMER_MMA_SYNC or SHKV_CONSUMER_TCGEN05: the consumer a decode
    call with this shape would run on this pool."""
    out = ctypes.c_int32()
    _check(load().shkv_decode_consumer(pool, n_models, hq, ctypes.byref(out)), "shkv_decode_consumer")
    return out.value


def shkv_tails_create(pool: int, cfg: shkv_tails_config) -> int:
    h = ctypes.c_void_p()
    _check(load().shkv_tails_create(pool, ctypes.byref(cfg), ctypes.byref(h)), "shkv_tails_create")
    return h.value


def shkv_tails_destroy(tails: int) -> None:
    _check(load().shkv_tails_destroy(tails), "shkv_tails_destroy")


def shkv_tails_set_lens(tails: int, batch: int, lens_ptr: int, stream: int) -> None:
    _check(load().shkv_tails_set_lens(tails, batch, lens_ptr, stream), "shkv_tails_set_lens")


def shkv_tails_get_lens(tails: int, batch: int, lens_ptr: int) -> None:
    _check(load().shkv_tails_get_lens(tails, batch, lens_ptr), "shkv_tails_get_lens")


def shkv_tails_append(tails: int, batch: int, n_new: int, k_new: int, v_new: int, stream: int) -> None:
    _check(load().shkv_tails_append(tails, batch, n_new, k_new, v_new, stream), "shkv_tails_append")


def shkv_decode_tails_workspace_size(pool: int, tails: int, batch: int, hq: int) -> int:
    n = ctypes.c_size_t()
    _check(load().shkv_decode_tails_workspace_size(pool, tails, batch, hq, ctypes.byref(n)),
           "shkv_decode_tails_workspace_size")
    return n.value


def shkv_decode_attention_tails(pool: int, tails: int, batch: int, hq: int, q: int, scale: float, out: int,
                                lse_out: int, workspace: int, workspace_bytes: int, stream: int) -> None:
    _check(load().shkv_decode_attention_tails(pool, tails, batch, hq, q, scale, out, lse_out, workspace,
                                              workspace_bytes, stream), "shkv_decode_attention_tails")


def shkv_pages_create(num_pages: int, page_size: int) -> int:
    h = ctypes.c_void_p()
    _check(load().shkv_pages_create(num_pages, page_size, ctypes.byref(h)), "shkv_pages_create")
    return h.value


def shkv_pages_destroy(pages: int) -> None:
    _check(load().shkv_pages_destroy(pages), "shkv_pages_destroy")


def shkv_prefill_attention(pool: int, batch: int, n_new: int, hq: int, q: int, scale: float, out: int,
                           lse_out: int, stream: int) -> None:
    _check(load().shkv_prefill_attention(pool, batch, n_new, hq, q, scale, out, lse_out, stream),
           "shkv_prefill_attention")
