"""GB300-native forward pass of causal Continuous Softmax Attention.

The compute lives in ``libcsa.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/csa.h``).  This package is the thin ctypes
binding over that library; nothing here computes attention.  Calls fail
loudly when the library has not been built.
"""
from .inputs import ZERO, COPY_FIRST, GIVEN  # noqa: F401

__all__ = ["ZERO", "COPY_FIRST", "GIVEN"]
