"""Paged decode attention over a block-paged KV cache, for one GB300 GPU.

The compute lives in ``libpkv.so`` (hand-written sm_103a CUDA behind the C ABI
declared in ``include/pkv.h``).  ``paged_decode_attention_cache_gb300.ops``
binds it for torch tensors; importing this package does not load the library.
"""
__all__ = ["ops", "workloads", "bytes_model"]
