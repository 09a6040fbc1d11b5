"""Attention over a paged KV cache for GB300 (sm_103a).

The compute path is ``libpkv.so`` (hand-written CUDA behind a C ABI, declared
in ``include/pkv.h``); ``paged_kv_cache_246_gb300.binding`` is its thin
ctypes binding.  Importing this package loads nothing: ``binding`` loads the
library on first use and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
