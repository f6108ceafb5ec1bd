"""GB300 (sm_103a) KV-cache page codec: FP8 E4M3FN, TurboQuant-style K, uniform V.

The codec itself is the C-ABI library ``libkvcodec.so`` built from ``csrc/``
(hand-written CUDA kernels plus a small host library); ``codec`` is its thin
ctypes binding and ``synth`` makes seeded synthetic KV caches.  Importing the
package does not load the library; the first codec call does, and fails with a
clear error when it has not been built.
"""
__all__ = ["codec", "synth"]
