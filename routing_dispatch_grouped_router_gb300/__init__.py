"""Deterministic MoE layer (router, dispatch, grouped SwiGLU GEMMs, combine;
forward and backward) for one GB300, behind the C ABI declared in include/mok.h.

The compute runs only in the CUDA library ``libmok.so`` built from ``csrc/``;
this package marshals arguments.  There is no CPU fallback: calls fail loudly
when the library is missing.
"""
