"""GPU-resident suffix-decoding drafter for GB300 (sm_103a).

The work runs in libsgd (hand-written CUDA behind the C ABI of
include/sgd.h); this package holds the ctypes binding, the build step and the
seeded workload generators.
"""
from .drafter import Proposal, SuffixDrafter  # noqa: F401
from . import _lib  # noqa: F401

__all__ = ["SuffixDrafter", "Proposal"]
