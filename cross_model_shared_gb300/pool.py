"""PyTorch-facing helpers over the libshkv C ABI.

PyTorch provides device memory and streams only; every step of the decode
path runs in libshkv's CUDA kernels.  ``SharedKVPool`` owns the torch tensors
the pool description points at (the paged K/V cache of PrefillShare
Sec. 3.3, shared by all decoders as in ICaRus key design 2) and forwards to
the C entry points.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np
import torch

from . import _native as N


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _require(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class SharedKVPool:
    """One paged KV cache shared by N decoders.

    k_pages / v_pages: bf16 [num_pages, num_kv_heads, page_size, head_dim]
    block_table: int32 [max_batch, max_pages_per_seq] (fill it, then call
    ``sync_block_table`` is not needed: the kernels read it in place)
    seq_lens: int32 [max_batch], owned by the pool after creation.
    """

    def __init__(self, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int,
                 max_batch: int, max_pages_per_seq: int, device=None,
                 k_pages: Optional[torch.Tensor] = None, v_pages: Optional[torch.Tensor] = None,
                 initial_seq_lens=None):
        N.load()
        device = torch.device(device if device is not None else "cuda")
        shape = (num_pages, num_kv_heads, page_size, head_dim)
        self.k_pages = k_pages if k_pages is not None else torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.v_pages = v_pages if v_pages is not None else torch.zeros(shape, dtype=torch.bfloat16, device=device)
        for name, t in (("k_pages", self.k_pages), ("v_pages", self.v_pages)):
            _require(t, torch.bfloat16, name)
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} shape {tuple(t.shape)} != {shape}")
        self.block_table = torch.full((max_batch, max_pages_per_seq), -1, dtype=torch.int32, device=device)
        self.seq_lens = torch.zeros(max_batch, dtype=torch.int32, device=device)
        self.error_word = torch.zeros(1, dtype=torch.int32, device=device)
        self.num_pages, self.page_size, self.num_kv_heads, self.head_dim = shape[0], page_size, num_kv_heads, head_dim
        self.max_batch, self.max_pages_per_seq = max_batch, max_pages_per_seq
        init = None
        if initial_seq_lens is not None:
            init = np.zeros(max_batch, dtype=np.int32)
            init[: len(initial_seq_lens)] = np.asarray(initial_seq_lens, dtype=np.int32)
        cfg = N.shkv_pool_config(
            num_pages=num_pages, page_size=page_size, num_kv_heads=num_kv_heads, head_dim=head_dim,
            max_batch=max_batch, max_pages_per_seq=max_pages_per_seq,
            k_pages=self.k_pages.data_ptr(), v_pages=self.v_pages.data_ptr(),
            block_table=self.block_table.data_ptr(), seq_lens=self.seq_lens.data_ptr(),
            error_word=self.error_word.data_ptr(),
            initial_seq_lens=init.ctypes.data if init is not None else None)
        torch.cuda.synchronize(device)
        self.handle = N.shkv_pool_create(cfg)
        self._workspace: Optional[torch.Tensor] = None

    # -- lifecycle ----------------------------------------------------------
    def close(self):
        if getattr(self, "handle", None):
            N.shkv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- lengths --------------------------------------------------------------
    def set_seq_lens(self, lens, stream=None):
        arr = np.ascontiguousarray(lens, dtype=np.int32)
        N.shkv_pool_set_seq_lens(self.handle, len(arr), arr.ctypes.data, _stream_ptr(stream))

    def host_seq_lens(self, batch: Optional[int] = None) -> np.ndarray:
        batch = self.max_batch if batch is None else batch
        out = np.zeros(batch, dtype=np.int32)
        N.shkv_pool_get_seq_lens(self.handle, batch, out.ctypes.data)
        return out

    # -- the path -------------------------------------------------------------
    def append_kv(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Partial-prefill append of [B, T, Hkv, D] bf16 K/V (PrefillShare Sec. 3.3)."""
        _require(k_new, torch.bfloat16, "k_new")
        _require(v_new, torch.bfloat16, "v_new")
        B, T, H, D = k_new.shape
        if tuple(v_new.shape) != (B, T, H, D) or H != self.num_kv_heads or D != self.head_dim:
            raise ValueError("k_new/v_new must be [B, T, num_kv_heads, head_dim]")
        N.shkv_append_kv(self.handle, B, T, k_new.data_ptr(), v_new.data_ptr(), _stream_ptr(stream))

    def workspace(self, batch: int, n_models: int, hq: int) -> torch.Tensor:
        need = N.shkv_decode_workspace_size(self.handle, batch, n_models, hq)
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = torch.zeros(need, dtype=torch.uint8, device=self.k_pages.device)
        return self._workspace

    def decode_attention(self, q: torch.Tensor, n_models: int, scale: Optional[float] = None,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         return_lse: bool = False, stream=None):
        """Stacked decode attention (ICaRus key design 3).

        q: bf16 [B, n_models * hq, head_dim], model-major.  Returns out (bf16,
        same shape) and, if asked, lse (fp32 [B, n_models * hq]).
        """
        _require(q, torch.bfloat16, "q")
        B, rows, D = q.shape
        if rows % n_models or D != self.head_dim:
            raise ValueError("q must be [B, n_models * hq, head_dim]")
        hq = rows // n_models
        if scale is None:
            scale = 1.0 / float(np.sqrt(D))
        if out is None:
            out = torch.empty_like(q)
        _require(out, torch.bfloat16, "out")
        if return_lse and lse is None:
            lse = torch.empty((B, rows), dtype=torch.float32, device=q.device)
        ws = self.workspace(B, n_models, hq)
        N.shkv_decode_attention(self.handle, B, n_models, hq, q.data_ptr(), float(scale), out.data_ptr(),
                                lse.data_ptr() if lse is not None else None, ws.data_ptr(), ws.numel(),
                                _stream_ptr(stream))
        return (out, lse) if (return_lse or lse is not None) else out

    _CONSUMERS = {"auto": N.SHKV_CONSUMER_AUTO, "mma": N.SHKV_CONSUMER_MMA_SYNC, "mma.sync": N.SHKV_CONSUMER_MMA_SYNC,
                  "umma": N.SHKV_CONSUMER_TCGEN05, "tcgen05": N.SHKV_CONSUMER_TCGEN05}

    def set_decode_consumer(self, consumer: str = "auto") -> None:
        """Name the decode consumer kernel of this pool: 'auto' (default),
        'mma' / 'mma.sync', or 'umma' / 'tcgen05' (taken where the shape
        allows it)."""
        if consumer not in self._CONSUMERS:
            raise ValueError(f"unknown consumer {consumer!r}")
        N.shkv_pool_set_decode_consumer(self.handle, self._CONSUMERS[consumer])

    def decode_consumer(self, n_models: int, hq: int) -> str:
        """'tcgen05' or 'mma.sync': the consumer kernel decode_attention runs
        for this shape on this pool."""
        c = N.shkv_decode_consumer(self.handle, n_models, hq)
        return "tcgen05" if c == N.SHKV_CONSUMER_TCGEN05 else "mma.sync"

    def prefill_attention(self, q: torch.Tensor, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                          lse: Optional[torch.Tensor] = None, return_lse: bool = False, stream=None):
        """Causal attention of the n_new tokens just appended (PrefillShare
        Sec. 3.3 partial prefill): q bf16 [B, n_new, hq, head_dim]; new token
        i attends the cached prefix and the new tokens up to itself."""
        _require(q, torch.bfloat16, "q")
        B, T, H, D = q.shape
        if D != self.head_dim:
            raise ValueError("q must be [B, n_new, hq, head_dim]")
        if scale is None:
            scale = 1.0 / float(np.sqrt(D))
        if out is None:
            out = torch.empty_like(q)
        _require(out, torch.bfloat16, "out")
        if return_lse and lse is None:
            lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
        N.shkv_prefill_attention(self.handle, B, T, H, q.data_ptr(), float(scale), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, _stream_ptr(stream))
        return (out, lse) if (return_lse or lse is not None) else out

    def check_errors(self, stream=None) -> int:
        """Synchronize and return (then clear) the device error bits."""
        return N.shkv_check_errors(self.handle, _stream_ptr(stream))


class DecoderTails:
    """Per-decoder unique tails over a SharedKVPool's pages (PrefillShare
    Sec. 3.3-4, Eqs. 8-9: each decoder extends the shared base cache with its
    own generated tokens; decoder m attends [shared prefix ++ its tail]).

    block_table: int32 [max_batch, n_models, max_tail_pages] (fill it with
    page indices of the shared pool; unused entries -1)
    tail_lens: int32 [max_batch, n_models], owned by the tails after creation.
    """

    def __init__(self, pool: SharedKVPool, max_batch: int, n_models: int, max_tail_pages: int,
                 initial_tail_lens=None):
        self.pool = pool
        dev = pool.k_pages.device
        self.max_batch, self.n_models, self.max_tail_pages = max_batch, n_models, max_tail_pages
        self.block_table = torch.full((max_batch, n_models, max_tail_pages), -1, dtype=torch.int32, device=dev)
        self.tail_lens = torch.zeros((max_batch, n_models), dtype=torch.int32, device=dev)
        init = None
        if initial_tail_lens is not None:
            init = np.zeros((max_batch, n_models), dtype=np.int32)
            t = np.asarray(initial_tail_lens, dtype=np.int32)
            init[: t.shape[0]] = t
        cfg = N.shkv_tails_config(max_batch=max_batch, n_models=n_models, max_tail_pages=max_tail_pages,
                                  block_table=self.block_table.data_ptr(), tail_lens=self.tail_lens.data_ptr(),
                                  initial_tail_lens=init.ctypes.data if init is not None else None)
        torch.cuda.synchronize(dev)
        self.handle = N.shkv_tails_create(pool.handle, cfg)
        self._workspace: Optional[torch.Tensor] = None

    def close(self):
        if getattr(self, "handle", None):
            N.shkv_tails_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_lens(self, lens, stream=None):
        arr = np.ascontiguousarray(lens, dtype=np.int32)
        N.shkv_tails_set_lens(self.handle, arr.shape[0], arr.ctypes.data, _stream_ptr(stream))

    def host_lens(self, batch: Optional[int] = None) -> np.ndarray:
        batch = self.max_batch if batch is None else batch
        out = np.zeros((batch, self.n_models), dtype=np.int32)
        N.shkv_tails_get_lens(self.handle, batch, out.ctypes.data)
        return out

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Append [B, N, T, Hkv, D] bf16 K/V to every decoder's tail."""
        _require(k_new, torch.bfloat16, "k_new")
        _require(v_new, torch.bfloat16, "v_new")
        B, M, T, H, D = k_new.shape
        if tuple(v_new.shape) != (B, M, T, H, D) or M != self.n_models:
            raise ValueError("k_new/v_new must be [B, n_models, T, num_kv_heads, head_dim]")
        N.shkv_tails_append(self.handle, B, T, k_new.data_ptr(), v_new.data_ptr(), _stream_ptr(stream))

    def workspace(self, batch: int, hq: int) -> torch.Tensor:
        need = N.shkv_decode_tails_workspace_size(self.pool.handle, self.handle, batch, hq)
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = torch.zeros(need, dtype=torch.uint8, device=self.pool.k_pages.device)
        return self._workspace

    def decode_attention(self, q: torch.Tensor, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                         lse: Optional[torch.Tensor] = None, return_lse: bool = False, stream=None):
        """Stacked decode where decoder m of request b attends the shared
        prefix and its own tail.  q: bf16 [B, n_models * hq, head_dim]."""
        _require(q, torch.bfloat16, "q")
        B, rows, D = q.shape
        if rows % self.n_models or D != self.pool.head_dim:
            raise ValueError("q must be [B, n_models * hq, head_dim]")
        hq = rows // self.n_models
        if scale is None:
            scale = 1.0 / float(np.sqrt(D))
        if out is None:
            out = torch.empty_like(q)
        _require(out, torch.bfloat16, "out")
        if return_lse and lse is None:
            lse = torch.empty((B, rows), dtype=torch.float32, device=q.device)
        ws = self.workspace(B, hq)
        N.shkv_decode_attention_tails(self.pool.handle, self.handle, B, hq, q.data_ptr(), float(scale),
                                      out.data_ptr(), lse.data_ptr() if lse is not None else None, ws.data_ptr(),
                                      ws.numel(), _stream_ptr(stream))
        return (out, lse) if (return_lse or lse is not None) else out


class PrefixPages:
    """Host-side refcounted page bookkeeping for a pool of ``num_pages``
    pages of ``page_size`` tokens (libshkv's page manager): reusable
    prefix-cache blocks, keyed by their token ids and shared across requests
    and decoder models, and transfer pages for one handoff (PrFaaS hybrid
    prefix cache pool; ICaRus key design 2)."""

    def __init__(self, num_pages: int, page_size: int):
        N.load()
        self.page_size = page_size
        self.handle = N.shkv_pages_create(num_pages, page_size)

    def close(self):
        if getattr(self, "handle", None):
            N.shkv_pages_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def acquire(self, tokens) -> Tuple[np.ndarray, int]:
        """(pages for the prompt, tokens already cached)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        npg = (len(t) + self.page_size - 1) // self.page_size
        out = np.zeros(max(1, npg), dtype=np.int32)
        hit = ctypes.c_int32()
        N._check(N.load().shkv_pages_acquire(self.handle, t.ctypes.data if len(t) else None, len(t),
                                             out.ctypes.data, npg, ctypes.byref(hit)), "shkv_pages_acquire")
        return out[:npg].copy(), hit.value

    def publish(self, tokens, pages) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        pg = np.ascontiguousarray(pages, dtype=np.int32)
        N._check(N.load().shkv_pages_publish(self.handle, t.ctypes.data if len(t) else None, len(t),
                                             pg.ctypes.data if len(pg) else None), "shkv_pages_publish")

    def release(self, pages) -> None:
        pg = np.ascontiguousarray(pages, dtype=np.int32)
        N._check(N.load().shkv_pages_release(self.handle, pg.ctypes.data if len(pg) else None, len(pg)),
                 "shkv_pages_release")

    def alloc_transfer(self, n: int) -> np.ndarray:
        out = np.zeros(max(1, n), dtype=np.int32)
        N._check(N.load().shkv_pages_alloc_transfer(self.handle, n, out.ctypes.data), "shkv_pages_alloc_transfer")
        return out[:n].copy()

    def stats(self) -> dict:
        info = N.shkv_pages_info()
        N._check(N.load().shkv_pages_stats(self.handle, ctypes.byref(info)), "shkv_pages_stats")
        return {f: getattr(info, f) for f, _ in info._fields_}

    def refcount(self, page: int) -> int:
        c = ctypes.c_int32()
        N._check(N.load().shkv_pages_refcount(self.handle, page, ctypes.byref(c)), "shkv_pages_refcount")
        return c.value


def splitkv_merge(o_part: torch.Tensor, lse_part: torch.Tensor, out: Optional[torch.Tensor] = None,
                  lse_out: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Log-sum-exp merge of split partials: o_part fp32 [S, B, rows, D],
    lse_part fp32 [S, B, rows] -> (bf16 [B, rows, D], fp32 [B, rows])."""
    _require(o_part, torch.float32, "o_part")
    _require(lse_part, torch.float32, "lse_part")
    S, B, rows, D = o_part.shape
    if out is None:
        out = torch.empty((B, rows, D), dtype=torch.bfloat16, device=o_part.device)
    if lse_out is None:
        lse_out = torch.empty((B, rows), dtype=torch.float32, device=o_part.device)
    N.shkv_splitkv_merge(S, B, rows, D, o_part.data_ptr(), lse_part.data_ptr(), out.data_ptr(),
                         lse_out.data_ptr(), _stream_ptr(stream))
    return out, lse_out
