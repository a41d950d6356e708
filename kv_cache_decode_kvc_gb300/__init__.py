"""GB300-native single-token KV-cache decode step.

The compute path is the CUDA library ``libkvc.so`` (built from ``csrc/``) behind the
C ABI declared in ``include/kvc.h``; :mod:`kv_cache_decode_kvc_gb300.kvc` is its thin
ctypes binding.  :mod:`kv_cache_decode_kvc_gb300.synth` holds the seeded input
generators.  Importing this package loads nothing; the binding loads the library on
first use and raises if it is missing.
"""
__all__ = ["kvc", "synth"]
