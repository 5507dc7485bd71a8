"""Persistent KV cache for GB300: append/evict and grouped-query attention.

The CUDA library (``libkvc.so``) is loaded on first use; see ``kvc`` for the
Python binding of its C ABI.
"""
