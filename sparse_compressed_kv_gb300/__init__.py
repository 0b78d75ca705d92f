"""GB300-native compressed sparse attention (CSA) decode.

The compute lives in ``libcsa.so`` (hand-written CUDA for sm_103a, C ABI in
``include/csa.h``); ``csa`` is its ctypes binding.
"""
from . import csa  # noqa: F401

__all__ = ["csa"]
