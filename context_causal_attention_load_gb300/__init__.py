"""Load-balanced context-parallel causal attention and GQA decode for GB300.

The compute lives in ``libcpattn.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/cpattn.h``); ``cpattn`` is a thin ctypes binding.
"""
