"""GB300 (sm_103a) sparse-attention decode path: DSA indexer + Top-K, GPU
hot-cache gather over a pinned host mirror, Q8G64 dequant, absorbed-MLA
attention, and append with batched write-back.

The compute lives in ``libdsa_decode.so`` (hand-written CUDA, C ABI in
``include/dsa_decode.h``); ``abi`` binds it with ctypes under the same names.
Importing this package does not load the library; the first call does, and it
raises if the library is missing.
"""
from . import abi  # noqa: F401

__all__ = ["abi"]
