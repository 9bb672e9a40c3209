"""Fused grouped-query attention over a KV cache, native to GB300 (sm_103a).

The compute runs in the CUDA library ``libgqa_attn.so`` built from ``csrc/``;
this package is a thin ctypes binding over its C ABI (see ``binding``).
Importing the package does not load the library; the first call does, and
fails loudly if it has not been built.
"""
