"""B300-native Attention-Aware Transform Coding (AATC) for KV caches.

The compute path lives in the CUDA library ``libaatc.so`` (sources in
``csrc/``, C ABI in ``include/aatc.h``); ``aatc`` is its thin ctypes binding.
Importing this package does not load the library; ``aatc.lib()`` does, and
fails loudly if it is missing.
"""
__all__ = ["aatc", "synth"]
