"""Quantized KV cache (KIVI / InnerQ style, 2/4-bit) with fused decode
attention over the packed cache, for GB300 (sm_103a).

The compute path is the C-ABI library ``libkvq`` (hand-written CUDA); the
Python binding in :mod:`bit_kv_cache_14_gb300.kvq` only marshals arguments.
Importing this package loads nothing; the library is loaded on first use and
raises if it has not been built.
"""
__all__ = ["kvq", "synth"]
