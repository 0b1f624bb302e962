"""Fused Mixture-of-Experts forward for GB300 (sm_103a).

The compute lives in ``libmoe.so`` (hand-written CUDA kernels behind the C ABI
of ``include/moe.h``); ``_lib`` is its ctypes binding and ``inputs`` the
seeded synthetic workloads.  Importing this package loads nothing; the first
call into ``_lib`` loads the library and raises if it is missing."""
from . import inputs  # noqa: F401

__all__ = ["inputs"]
