"""Sparse Mixture-of-Experts layer forward pass on one B300 (sm_103a).

The compute lives in ``libmoe_b300.so`` (hand-written CUDA kernels behind a C ABI, declared in
``include/moe_b300.h``).  ``binding`` is the thin ctypes layer over it; ``inputs`` draws the seeded
synthetic workloads.  Importing this package loads nothing; ``binding`` loads the library on first use
and raises if it is missing.
"""
