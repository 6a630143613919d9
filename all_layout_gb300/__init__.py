"""GB300-native fused attention + Ulysses post-attention All-to-All layout.

The compute path is the C-ABI library ``libxs.so`` (CUDA for sm_103a, built
from ``csrc/``); ``all_layout_gb300.xs`` is its thin ctypes binding. Importing
this package does not load the library; ``all_layout_gb300.xs`` does, and it
raises if the library is missing.
"""
__all__ = ["inputs", "xs"]
