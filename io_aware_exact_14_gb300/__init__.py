"""GB300-native exact attention: tiled forward with online softmax, recompute backward.

The compute path is the C-ABI library ``libfa.so`` (hand-written sm_103a
kernels); ``io_aware_exact_14_gb300.fa`` is a thin ctypes binding over it.
Importing this package does not load the library; the first call does, and
raises if the library or a CUDA device is missing.
"""
__all__ = ["fa", "workloads", "counts"]
