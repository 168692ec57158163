"""VerKV on GB300: KVFetch verified attention over a PoissonComp-compressed KV cache.

The compute path is the C-ABI library ``libverkv.so`` (hand-written CUDA for
sm_103a, built from ``csrc/``); ``verified_kv_cache_gb300.binding`` is the thin
ctypes layer over it.  Importing this package does not load the library.
"""
__all__ = ["binding", "workloads", "build"]
