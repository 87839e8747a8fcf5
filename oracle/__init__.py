"""fp64 CPU oracle for shared-KV multi-decoder paged decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  The
library path never imports this package, and this package never imports the
library: the two share no code.

The arithmetic lives in ``shkv_oracle.c`` (plain C, fp64, pthreads); this
module only builds it with gcc and marshals numpy arrays to it.  Each wrapper
names the passage the C function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "shkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_shkv.so")
_lock = threading.Lock()
_lib = None

INT_MAX = 2**31 - 1
_errors = {1: "invalid argument", 2: "page index outside the pool", 3: "out of memory"}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math: IEEE fp64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_decode_attention.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P,
                                                    ctypes.c_int32, ctypes.c_int32,
                                                    ctypes.c_double, P, P, i]
            lib.oracle_decode_attention.restype = i
            lib.oracle_decode_attention_tails.argtypes = [i, i, i, i, i, i, i, i, i, P, P, P, P, P, P, P,
                                                          ctypes.c_double, P, P, i]
            lib.oracle_decode_attention_tails.restype = i
            lib.oracle_prefill_attention.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, ctypes.c_double, P, P, i]
            lib.oracle_prefill_attention.restype = i
            lib.oracle_splitkv_merge.argtypes = [i, i, i, i, P, P, P, P]
            lib.oracle_splitkv_merge.restype = i
            lib.oracle_append_kv.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P]
            lib.oracle_append_kv.restype = i
            lib.oracle_gather_kv.argtypes = [i, i, i, i, i, i, P, P, P, P]
            lib.oracle_gather_kv.restype = i
            lib.oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(st: int, what: str):
    if st != 0:
        raise RuntimeError(f"oracle {what}: {_errors.get(st, st)}")


def num_threads() -> int:
    return _load().oracle_num_threads()


def decode_attention(q, k_pages, v_pages, block_table, seq_lens, *, n_models: int,
                     hq: int, scale: float, t_begin: int = 0, t_end: int = INT_MAX,
                     nthreads: int = 0):
    """Attention of N stacked decoders over one shared paged KV cache.

    Follows ICaRus key designs 2-3 (one identical cache, queries concatenated
    along heads) over PrefillShare's paged KV blocks.  ``q`` is bf16 bits
    [B, N*Hq, D]; pools are bf16 bits [num_pages, Hkv, P, D].  Returns fp64
    (out [B, N*Hq, D], lse [B, N*Hq]).  A token window [t_begin, t_end) gives
    the partial attention of a split.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, rows, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    assert D2 == D and rows == n_models * hq and bt.shape[0] >= B
    out = np.zeros((B, rows, D), dtype=np.float64)
    lse = np.zeros((B, rows), dtype=np.float64)
    st = _load().oracle_decode_attention(B, n_models, hq, Hkv, D, P, num_pages, bt.shape[1],
                                         _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(bt),
                                         _ptr(lens), int(t_begin), int(t_end), float(scale),
                                         _ptr(out), _ptr(lse), int(nthreads))
    _check(st, "decode_attention")
    return out, lse


def decode_attention_tails(q, k_pages, v_pages, block_table, seq_lens, tail_table, tail_lens, *,
                           n_models: int, hq: int, scale: float, nthreads: int = 0):
    """Stacked decode where each decoder also attends its own unique tail.

    Follows PrefillShare Sec. 3.3-4 (decode starts from the shared base cache
    and extends it with the decoder's own Delta C_t; Eqs. 8-9 store the shared
    prefix once and N unique tails).  Decoder m of request b attends the
    concatenation of the shared tokens [0, L_b) and its tail tokens
    [0, T_{b,m}).  ``tail_table`` is int32 [B, N, max_tail_pages] and
    ``tail_lens`` int32 [B, N], into the same page pool.  Returns fp64
    (out [B, N*Hq, D], lse [B, N*Hq]).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    tt = np.ascontiguousarray(tail_table, dtype=np.int32)
    tl = np.ascontiguousarray(tail_lens, dtype=np.int32)
    B, rows, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    assert D2 == D and rows == n_models * hq and bt.shape[0] >= B
    assert tt.shape[:2] == (B, n_models) and tl.shape == (B, n_models)
    out = np.zeros((B, rows, D), dtype=np.float64)
    lse = np.zeros((B, rows), dtype=np.float64)
    st = _load().oracle_decode_attention_tails(B, n_models, hq, Hkv, D, P, num_pages, bt.shape[1], tt.shape[2],
                                               _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(bt), _ptr(lens),
                                               _ptr(tt), _ptr(tl), float(scale), _ptr(out), _ptr(lse),
                                               int(nthreads))
    _check(st, "decode_attention_tails")
    return out, lse


def prefill_attention(q, k_pages, v_pages, block_table, seq_lens, *, scale: float, nthreads: int = 0):
    """Causal attention of n_new appended tokens over the cached prefix and
    themselves (PrefillShare Sec. 3.3, partial prefill on a cache hit).

    ``q`` is bf16 bits [B, n_new, Hq, D]; ``seq_lens`` already include the
    n_new tokens, whose K/V are in the pool.  New token i of request b is at
    position seq_lens[b] - n_new + i and attends keys 0 .. its position.
    Returns fp64 (out [B, n_new, Hq, D], lse [B, n_new, Hq])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, T, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    assert D2 == D and bt.shape[0] >= B
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    lse = np.zeros((B, T, Hq), dtype=np.float64)
    st = _load().oracle_prefill_attention(B, T, Hq, Hkv, D, P, num_pages, bt.shape[1], _ptr(q), _ptr(k_pages),
                                          _ptr(v_pages), _ptr(bt), _ptr(lens), float(scale), _ptr(out), _ptr(lse),
                                          int(nthreads))
    _check(st, "prefill_attention")
    return out, lse


def splitkv_merge(o_part, lse_part):
    """Log-sum-exp merge of split partials (fp64).  o_part [S, B, rows, D],
    lse_part [S, B, rows] -> (out [B, rows, D], lse [B, rows])."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    S, B, rows, D = o_part.shape
    out = np.zeros((B, rows, D), dtype=np.float64)
    lse = np.zeros((B, rows), dtype=np.float64)
    _check(_load().oracle_splitkv_merge(S, B, rows, D, _ptr(o_part), _ptr(lse_part),
                                        _ptr(out), _ptr(lse)), "splitkv_merge")
    return out, lse


def append_kv(k_pages, v_pages, block_table, seq_lens, k_new, v_new):
    """Partial-prefill append (PrefillShare Sec. 3.3).  Returns new copies of
    (k_pages, v_pages, seq_lens); the inputs are left untouched."""
    k = np.array(k_pages, dtype=np.uint16, copy=True, order="C")
    v = np.array(v_pages, dtype=np.uint16, copy=True, order="C")
    lens = np.array(seq_lens, dtype=np.int32, copy=True, order="C")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    kn = np.ascontiguousarray(k_new, dtype=np.uint16)
    vn = np.ascontiguousarray(v_new, dtype=np.uint16)
    B, T, Hkv, D = kn.shape
    num_pages, _, P, _ = k.shape
    _check(_load().oracle_append_kv(B, T, Hkv, D, P, num_pages, bt.shape[1], _ptr(k), _ptr(v),
                                    _ptr(bt), _ptr(lens), _ptr(kn), _ptr(vn)), "append_kv")
    return k, v, lens


def gather_kv(pool, block_table, seq_lens, b: int):
    """Logical cache of request b through the block table: bf16 bits
    [L_b, Hkv, D]."""
    pool = np.ascontiguousarray(pool, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_pages, Hkv, P, D = pool.shape
    out = np.zeros((int(lens[b]), Hkv, D), dtype=np.uint16)
    _check(_load().oracle_gather_kv(int(b), Hkv, D, P, num_pages, bt.shape[1], _ptr(pool),
                                    _ptr(bt), _ptr(lens), _ptr(out)), "gather_kv")
    return out
