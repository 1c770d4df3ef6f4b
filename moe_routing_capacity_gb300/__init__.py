"""GB300 (sm_103a) implementation of the pooled-wave MoE layer forward.

The compute lives in ``libmoe_pooled_wave.so`` (hand-written CUDA behind a
C ABI, see ``include/moe_pooled_wave.h``); ``abi`` is its ctypes binding and
``layer`` a thin wrapper that owns device buffers (through PyTorch) and calls
the five entry points in order.  ``workloads`` draws the seeded synthetic
inputs.  Importing the package loads nothing; the library is loaded on first
use and its absence is an error.
"""
__all__ = ["abi", "layer", "workloads"]
