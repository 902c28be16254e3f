"""Exact IO-aware attention (FlashAttention-style forward with LSE, recompute backward)
for NVIDIA GB300 (sm_103a), behind a C ABI (``include/fa.h``).

The compute runs only in the CUDA library ``libfa.so`` built from ``csrc/``; this package
marshals arguments to it. There is no CPU fallback: every entry point raises if the
library is missing.
"""
