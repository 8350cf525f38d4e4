"""paged_kv_cache_143_gb300 — paged-KV attention hot path for one GB300 (sm_103a).

The compute runs in ``libpa.so`` (hand-written CUDA, C ABI declared in
``include/pa.h``). ``paged_kv_cache_143_gb300.pa`` is the thin binding that
passes torch device pointers and the current stream to it; the library is
loaded on first use and a missing or unbuildable library raises immediately
(there is no CPU fallback).
"""
__all__ = ["pa", "accounting"]
