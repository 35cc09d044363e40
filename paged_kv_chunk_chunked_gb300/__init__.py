"""Paged chunk attention for GB300 (sm_103a).

Causal GQA attention forward and backward for one query chunk against a paged
KV cache, with in-place fp32 dK/dV accumulation into a paged gradient pool, a
page-level top-K sparse variant and a pinned-host page streamer. The compute
runs in the C-ABI library ``libpkv.so`` (hand-written CUDA); ``binding`` is a
thin ctypes layer over it. Importing this package does not load the library;
``binding.lib()`` does, and fails loudly when it is missing.
"""
__version__ = "0.1.0"
