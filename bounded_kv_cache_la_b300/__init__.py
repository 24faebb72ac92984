"""Bounded-KV-cache chunk attention for streaming video DiTs on B300 (sm_103a).

The compute path is the C-ABI library liblacache.so (include/la_cache.h);
`capi` is its ctypes binding.  Build with `python -m bounded_kv_cache_la_b300.build`.
"""
from . import capi  # noqa: F401
