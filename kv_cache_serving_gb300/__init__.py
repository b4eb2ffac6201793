"""Diagonal-aware sparse decode attention over a paged KV cache, for GB300 (sm_103a).

The compute lives in the C-ABI library ``libdsa.so`` (hand-written CUDA, built
from ``csrc/``); ``kv_cache_serving_gb300.dsa`` is its thin ctypes binding and
``kv_cache_serving_gb300.workloads`` draws seeded synthetic inputs.  Importing
the package loads nothing: the library is opened on first use of ``dsa``.
"""
__all__ = ["dsa", "workloads"]
