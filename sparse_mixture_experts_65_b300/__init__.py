"""B300-native forward pass of one sparse top-k Mixture-of-Experts FFN layer.

The compute lives in libmoe.so (hand-written sm_103a CUDA behind the C ABI
in include/moe.h); this package holds its ctypes binding (``layer``), the
build script and the seeded synthetic workloads.  The shared library is
loaded on first use and its absence is an error: there is no fallback.
"""
from . import layer, workloads  # noqa: F401

__all__ = ["layer", "workloads"]
