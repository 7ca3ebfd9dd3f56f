"""GB300-native paged-KV decode attention with grouped-query heads.

The compute path is the C-ABI library ``libpagedkv.so`` (hand-written sm_103a
kernels, declared in ``include/pagedkv.h``); :mod:`.binding` is its thin
Python binding. :mod:`.workloads` and :mod:`.allocator` are host-side input
generation and block bookkeeping.

Importing the package does not load the CUDA library; ``binding`` does, and
raises if it is missing: there is no CPU fallback.
"""

__all__ = ["binding", "workloads", "allocator"]
