"""Sparse-MoE feed-forward layer (Step 3.5 Flash shape) on GB300 / sm_103a.

The compute path is the CUDA library ``libmoe.so`` built from ``csrc/``;
``binding`` is a thin ctypes layer over its C ABI (``include/moe.h``).
Importing this package does not load the library: the first call into
``binding`` does, and raises if it has not been built.
"""
__all__ = ["binding", "synth"]
