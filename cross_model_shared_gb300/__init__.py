"""Shared-KV multi-decoder paged decode attention for GB300 (sm_103a).

N task decoders that share one frozen prefill/encoder module read one paged
KV cache; their queries are stacked along the head axis so each KV page is
read from HBM once per decode step (ICaRus key design 3; PrefillShare
Sec. 3.3).  The compute path is libshkv (hand-written CUDA behind a C ABI,
``include/shkv.h``); this package is its Python binding.

Submodules load lazily so that the input generators (``workloads``) can be
imported without a GPU or a built library.
"""
import importlib

__all__ = ["SharedKVPool", "DecoderTails", "PrefixPages", "splitkv_merge", "native", "workloads", "build"]


def __getattr__(name):
    if name in ("SharedKVPool", "DecoderTails", "PrefixPages", "splitkv_merge"):
        return getattr(importlib.import_module(".pool", __name__), name)
    if name == "native":
        return importlib.import_module("._native", __name__)
    if name in ("workloads", "build"):
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
