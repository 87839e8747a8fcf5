"""Seeded synthetic inputs for shared-KV multi-decoder decode attention.

This module only *makes inputs*: request lengths, the paged pool's block
table, and bf16 query / key / value bits.  It holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can draw their inputs
from it without sharing any of the method.

Workload shapes follow the pages' model families and serving mixes:

* ICaRus (key design 3): N task decoders concatenate their queries along
  the head axis and attend one shared KV cache; serving runs used
  LLaMA-3.1-8B and Qwen3-8B/14B with 2, 4 and 8 models.
* PrefillShare (Sec. 3.3 / Sec. 7): the shared cache is held in vLLM-style
  KV blocks (pages); a returning session runs a partial prefill that appends
  new tokens to the cached prefix.
* PrFaaS (training/deployment setup): long-context request lengths follow
  a truncated log-normal with a mean of about 27K tokens.

Readings where the pages are silent (stated once here, used everywhere):
"1K"/"4K"/"27K" are multiples of 1024; the log-normal sigma is 1; the
log-normal mean for the Qwen3-8B mix is the untruncated mean, then rounded
and clipped; the 27K mix is truncated by rejection with mu calibrated so the
truncated mean is 27648.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict

import numpy as np

__all__ = [
    "Workload", "CONFIGS", "CONFIG_ORDER", "make_workload", "custom_workload",
    "bf16_bits_from_f32", "f32_from_bf16_bits", "gen_q", "gen_pool", "gen_append",
    "unique_kv_bytes", "pages_required", "trunc_lognormal_mu",
]


# ---------------------------------------------------------------------------
# bf16 bit helpers (input encoding only)
# ---------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even) and return
    the raw uint16 bit patterns.  Inputs are finite normal draws."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# workload description
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    """One decode-attention problem over a shared paged KV pool.

    Attributes are the pages' notation: ``B`` requests, ``N`` decoders,
    ``Hq`` query heads per decoder, ``Hkv`` KV heads, head dim ``D`` and page
    size ``P`` tokens.  ``lens_prefill`` are the cached lengths before any
    partial-prefill append, ``n_append`` the tokens appended per request, and
    ``lens_final`` the lengths attention runs over.
    """
    name: str
    B: int
    N: int
    Hq: int
    Hkv: int
    D: int
    P: int
    seed: int
    lens_prefill: np.ndarray
    n_append: int
    block_table: np.ndarray          # int32 [B, max_pages_per_seq], -1 = unused
    num_pages: int

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def R(self) -> int:
        """Stacked query rows per KV head (N decoders x GQA group)."""
        return self.N * self.G

    @property
    def rows(self) -> int:
        """Query rows per request: N * Hq, model-major."""
        return self.N * self.Hq

    @property
    def lens_final(self) -> np.ndarray:
        return (self.lens_prefill + self.n_append).astype(np.int32)

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def pages_per_request(self) -> np.ndarray:
        return (self.lens_final + self.P - 1) // self.P


# ---------------------------------------------------------------------------
# length mixes
# ---------------------------------------------------------------------------
def trunc_lognormal_mu(mean: float, sigma: float, lo: float, hi: float) -> float:
    """mu such that LogNormal(mu, sigma) conditioned on [lo, hi] has the given
    mean (closed form of the truncated log-normal mean, solved by bisection)."""
    from math import erf, exp, log, sqrt

    def phi(z):
        return 0.5 * (1.0 + erf(z / sqrt(2.0)))

    def tmean(mu):
        a, b = (log(lo) - mu) / sigma, (log(hi) - mu) / sigma
        num = phi(b - sigma) - phi(a - sigma)
        den = phi(b) - phi(a)
        return exp(mu + 0.5 * sigma * sigma) * num / den

    left, right = log(lo) - 5 * sigma, log(hi) + 5 * sigma
    for _ in range(200):
        mid = 0.5 * (left + right)
        if tmean(mid) < mean:
            left = mid
        else:
            right = mid
    return 0.5 * (left + right)


def _lengths(kind: str, B: int, rng: np.random.Generator, **kw) -> np.ndarray:
    if kind == "const":
        return np.full(B, kw["value"], dtype=np.int64)
    if kind == "uniform":
        return rng.integers(kw["lo"], kw["hi"] + 1, size=B, dtype=np.int64)
    if kind == "lognormal_clip":
        mu = math.log(kw["mean"]) - 0.5 * kw["sigma"] ** 2
        x = np.rint(rng.lognormal(mu, kw["sigma"], size=B))
        return np.clip(x, kw["lo"], kw["hi"]).astype(np.int64)
    if kind == "lognormal_trunc":
        mu = trunc_lognormal_mu(kw["mean"], kw["sigma"], kw["lo"], kw["hi"])
        out = []
        while len(out) < B:
            x = np.rint(rng.lognormal(mu, kw["sigma"], size=4 * B))
            x = x[(x >= kw["lo"]) & (x <= kw["hi"])]
            out.extend(int(v) for v in x[: B - len(out)])
        return np.asarray(out, dtype=np.int64)
    raise ValueError(f"unknown length mix {kind!r}")


# name -> (shape, length mix); seeds are the config index.
CONFIGS: Dict[str, dict] = {
    # tiny: 1 request, 2 decoders, 2 KV heads, GQA 4, d=64, 256 tokens, P=16
    "tiny": dict(B=1, N=2, Hq=8, Hkv=2, D=64, P=16, n_append=0, seed=0,
                 lens=dict(kind="const", value=256)),
    # Llama-3.1-8B attention, ICaRus encoder+decoder concat (N=2)
    "llama8b": dict(B=32, N=2, Hq=32, Hkv=8, D=128, P=16, n_append=0, seed=1,
                    lens=dict(kind="uniform", lo=1024, hi=8192)),
    # Qwen3-8B attention, 4 agent decoders
    "qwen8b": dict(B=64, N=4, Hq=32, Hkv=8, D=128, P=16, n_append=0, seed=2,
                   lens=dict(kind="lognormal_clip", mean=4096, sigma=1.0, lo=512, hi=32768)),
    # Qwen3-14B attention, 8 decoders, PrFaaS-style long mix (mean ~27K)
    "qwen14b": dict(B=128, N=8, Hq=40, Hkv=8, D=128, P=32, n_append=0, seed=3,
                    lens=dict(kind="lognormal_trunc", mean=27648, sigma=1.0, lo=1024, hi=65536)),
    # Qwen3-1.7B attention, 128K context + 512-token partial-prefill append
    "long": dict(B=4, N=8, Hq=16, Hkv=8, D=128, P=16, n_append=512, seed=4,
                 lens=dict(kind="const", value=131072)),
}
CONFIG_ORDER = ["tiny", "llama8b", "qwen8b", "qwen14b", "long"]


def _assign_pages(lens_final: np.ndarray, P: int, rng: np.random.Generator,
                  spare_pages: int = 0):
    """Give each request ceil(L/P) physical pages drawn from one random
    permutation of the pool (requests never share pages)."""
    pages = (lens_final + P - 1) // P
    total = int(pages.sum())
    num_pages = total + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = int(max(1, pages.max()))
    bt = np.full((len(lens_final), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[off: off + n]
        off += int(n)
    return bt, num_pages


def custom_workload(name: str, B: int, N: int, Hq: int, Hkv: int, D: int, P: int,
                    lens_prefill, n_append: int = 0, seed: int = 0,
                    spare_pages: int = 0, extra_pages_per_seq: int = 0) -> Workload:
    """A workload with explicit lengths (used for reduced-size and edge cases)."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    rng = np.random.default_rng(seed)
    lens_prefill = np.asarray(lens_prefill, dtype=np.int64)
    lens_final = lens_prefill + n_append
    bt, num_pages = _assign_pages(lens_final, P, rng, spare_pages)
    if extra_pages_per_seq:
        bt = np.concatenate([bt, np.full((B, extra_pages_per_seq), -1, np.int32)], axis=1)
    return Workload(name=name, B=B, N=N, Hq=Hq, Hkv=Hkv, D=D, P=P, seed=seed,
                    lens_prefill=lens_prefill.astype(np.int32), n_append=n_append,
                    block_table=bt, num_pages=num_pages)


def tails_spare_pages(tail_lens, P: int, reserve_tokens: int = 0) -> int:
    """Pages needed by per-decoder tails of the given lengths [B, N], each
    with room for ``reserve_tokens`` more."""
    t = np.asarray(tail_lens, dtype=np.int64) + reserve_tokens
    return int(((t + P - 1) // P).sum())


def make_tails(wl: Workload, tail_lens, seed: int = 0, reserve_tokens: int = 0, extra_pages_per_tail: int = 0):
    """Per-decoder unique tails (PrefillShare Eq. 9's N * L_unique) placed in
    the pool pages the shared requests do not use, in a seeded random order.

    ``tail_lens`` is [B, N] tokens; every tail gets pages for
    ``reserve_tokens`` more (room for appends) and the table
    ``extra_pages_per_tail`` unused (-1) entries.  Returns (tail_table int32
    [B, N, max_tail_pages], tail_lens int32 [B, N]).  The workload must have
    been made with enough spare pages (``tails_spare_pages``)."""
    tl = np.asarray(tail_lens, dtype=np.int64).reshape(wl.B, wl.N)
    used = set(int(x) for x in wl.block_table[wl.block_table >= 0].ravel())
    free = np.array([pg for pg in range(wl.num_pages) if pg not in used], dtype=np.int32)
    rng = np.random.default_rng(seed)
    free = free[rng.permutation(len(free))]
    pages = (tl + reserve_tokens + wl.P - 1) // wl.P
    need = int(pages.sum())
    if need > len(free):
        raise ValueError(f"tails need {need} pages, the pool has {len(free)} spare")
    width = int(max(1, pages.max())) + extra_pages_per_tail
    tt = np.full((wl.B, wl.N, width), -1, dtype=np.int32)
    off = 0
    for b in range(wl.B):
        for m in range(wl.N):
            n = int(pages[b, m])
            tt[b, m, :n] = free[off: off + n]
            off += n
    return tt, tl.astype(np.int32)


def make_workload(name: str, replica: int = 0) -> Workload:
    """The named configuration, seeded by its index.  ``replica`` r > 0 draws
    another batch of the same shape and length mix (seeded by the index and
    r), for a job whose global batch is several batches of the configuration."""
    c = CONFIGS[name]
    rng = np.random.default_rng(c["seed"] if replica == 0 else [c["seed"], 5005, replica])
    lens = _lengths(B=c["B"], rng=rng, **c["lens"])
    lens_final = lens + c["n_append"]
    bt, num_pages = _assign_pages(lens_final, c["P"], rng)
    return Workload(name=name, B=c["B"], N=c["N"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"],
                    P=c["P"], seed=c["seed"], lens_prefill=lens.astype(np.int32),
                    n_append=c["n_append"], block_table=bt, num_pages=num_pages)


# ---------------------------------------------------------------------------
# value generators (N(0,1) fp32 -> bf16 RNE), host side
# ---------------------------------------------------------------------------
def _normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_bits_from_f32(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def gen_q(wl: Workload, salt: int = 0) -> np.ndarray:
    """Stacked queries, bf16 bits [B, N*Hq, D], model-major rows."""
    rng = np.random.default_rng([wl.seed, 101, salt])
    return _normal_bf16(rng, (wl.B, wl.rows, wl.D))


def gen_pool(wl: Workload, salt: int = 0):
    """K and V pages, bf16 bits [num_pages, Hkv, P, D] each.  Every slot is
    filled, including the unused tail slots of each request's last page, so
    masking errors show up as wrong values."""
    rng = np.random.default_rng([wl.seed, 202, salt])
    shape = (wl.num_pages, wl.Hkv, wl.P, wl.D)
    return _normal_bf16(rng, shape), _normal_bf16(rng, shape)


def gen_append(wl: Workload, salt: int = 0):
    """Partial-prefill K/V to append, bf16 bits [B, T, Hkv, D] each."""
    rng = np.random.default_rng([wl.seed, 303, salt])
    shape = (wl.B, wl.n_append, wl.Hkv, wl.D)
    return _normal_bf16(rng, shape), _normal_bf16(rng, shape)


# ---------------------------------------------------------------------------
# accounting (PrefillShare Eqs. 8-9)
# ---------------------------------------------------------------------------
def pages_required(lens, P: int, n_models: int, shared: bool) -> int:
    """KV pages needed to hold every request's context for ``n_models``
    decoders.  Shared (PrefillShare Eq. 9 with no per-model tail): one copy.
    Unshared (Eq. 8): one copy per model."""
    pages = int(((np.asarray(lens, dtype=np.int64) + P - 1) // P).sum())
    return pages if shared else n_models * pages


def unique_kv_bytes(wl: Workload) -> int:
    """Bytes of the distinct KV pages one decode step must read."""
    return int(wl.pages_per_request().sum()) * wl.P * wl.Hkv * wl.D * 2 * 2


# ---------------------------------------------------------------------------
# device-side value generator for pools too large to draw on the host
# ---------------------------------------------------------------------------
def gen_pool_device(wl: Workload, device="cuda", salt: int = 0, chunk: int = 1 << 28):
    """K and V pages drawn N(0,1) on the GPU with a seeded torch generator and
    rounded to bf16 (torch's fp32 -> bf16 cast rounds to nearest even).  Used
    for multi-GB pools; tests read back the pages they check."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(wl.seed) * 1000003 + 202 + int(salt))
    shape = (wl.num_pages, wl.Hkv, wl.P, wl.D)
    out = []
    for _ in range(2):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        for s in range(0, flat.numel(), chunk):
            e = min(flat.numel(), s + chunk)
            flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        out.append(t)
    return out[0], out[1]
