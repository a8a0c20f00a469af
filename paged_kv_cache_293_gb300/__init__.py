"""GB300-native paged KV-cache decode.

The kernels live in ``csrc/`` behind a C-ABI shared library (``libpagedkv.so``,
declared in ``include/pagedkv.h``).  ``paged_kv_cache_293_gb300.pagedkv`` is the
thin ctypes binding with the same entry-point names; importing it fails loudly
when the library has not been built.  ``workloads`` draws seeded synthetic
inputs and ``accounting`` holds the byte / flop counts used for rooflines.
"""
__all__ = ["pagedkv", "workloads", "accounting"]
