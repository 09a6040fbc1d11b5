"""fp64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``.  The
library (``paged_kv_cache_246_gb300``) never imports it, and it imports
nothing from the library: the two share no code.
"""
from .paged_attention import *  # noqa: F401,F403
