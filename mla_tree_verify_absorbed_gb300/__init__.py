"""DDTree verify attention, MLA in absorbed form, for GB300 (sm_103a).

The compute path is a C-ABI CUDA library (``lib/libmla_verify.so``, built from
``csrc/``); ``api`` is a thin ctypes binding over it.  Importing this package
does not load the library: ``api`` loads it on first use and raises when it is
missing, so there is no silent fallback.
"""
__all__ = ["inputs", "api"]
