"""GB300 (sm_103a) decode-time KV-cache compression event.

The computation lives in ``libkvc.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/kvc.h``). ``eviction_gb300.kvc`` is a thin ctypes binding
with the same entry-point names that takes torch tensors and passes their device
pointers and the current CUDA stream. There is no CPU fallback: every call fails
loudly if the library or a CUDA device is missing.
"""
from .kvc import (ABLATIONS, Config, Handle, KvcError, library_path, load_library,  # noqa: F401
                  mass_noalloc, ENTRY_POINTS)

__all__ = ["ABLATIONS", "Config", "Handle", "KvcError", "library_path", "load_library",
           "mass_noalloc", "ENTRY_POINTS"]
