"""Exact IO-aware attention (forward + backward) for GB300 (sm_103a).

The compute lives in a C-ABI shared library (``libfa_gb300.so``, see
``include/fa.h``); :mod:`exact_io_aware_28_gb300.fa` is the thin ctypes binding
with the same names as the C entry points.  :mod:`.workloads` draws the seeded
synthetic inputs and :mod:`.accounting` holds the FLOP/byte conventions.
"""
__all__ = ["fa", "workloads", "accounting"]
