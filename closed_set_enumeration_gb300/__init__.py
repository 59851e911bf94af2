"""GB300-native formal-concept enumeration (Close-by-One with saturation pruning).

The work runs in ``libfca.so`` (CUDA, sm_103a) behind the C ABI of
``include/fca.h``; :mod:`closed_set_enumeration_gb300.fca` is its ctypes
binding and :mod:`closed_set_enumeration_gb300.contexts` draws the seeded
synthetic contexts. Build the library with
:func:`closed_set_enumeration_gb300.build.build`.
"""
__all__ = ["build", "contexts", "fca"]
