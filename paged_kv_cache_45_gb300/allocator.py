"""Host-side physical block allocator for the paged KV pool.

A free list plus a per-block reference count. Block 0 is never handed out:
it is kept for health checks, as TGI's router allocator does ("text-generation-
inference" on pyshine, section "The radix prefix cache"). Blocks return to the
free list when their last reference is dropped ("How to Speed Up LLM Inference:
KV Cache to Production Serving", section "Architecture: inside a modern
inference engine": finished sequences release their KV blocks), exactly once
("The inference request lifecycle", section "Every transition needs an owner
and a release rule").

This is scheduler bookkeeping on the host; the device kernels only ever see
the resulting block tables and slot mappings.
"""

from __future__ import annotations

import numpy as np


class PoolExhausted(RuntimeError):
    """Raised when an allocation asks for more blocks than are free."""


class BlockAllocator:
    """Free list + refcounts over ``num_blocks`` physical blocks.

    ``order`` (optional) fixes the order blocks leave the free list, which is
    how the workloads shuffle physical placement with a seeded permutation.
    """

    def __init__(self, num_blocks: int, order=None, reserve_block0: bool = True):
        if num_blocks < 2 and reserve_block0:
            raise ValueError("a pool needs at least block 0 plus one usable block")
        self.num_blocks = int(num_blocks)
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)
        first = 1 if reserve_block0 else 0
        ids = np.arange(first, self.num_blocks) if order is None else np.asarray(order)
        ids = [int(i) for i in ids if int(i) >= first]
        if sorted(ids) != list(range(first, self.num_blocks)):
            raise ValueError("order must be a permutation of the usable block ids")
        # pop() takes from the end: reverse so blocks leave in `order`
        self._free = ids[::-1]
        self.reserved = 0 if reserve_block0 else None

    # -- queries -----------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._free)

    def owned(self) -> np.ndarray:
        return np.nonzero(self.refcount > 0)[0]

    # -- operations ----------------------------------------------------------
    def allocate(self, n: int) -> list[int]:
        if n > len(self._free):
            raise PoolExhausted(f"asked for {n} blocks, {len(self._free)} free")
        out = [self._free.pop() for _ in range(n)]
        for b in out:
            assert self.refcount[b] == 0
            self.refcount[b] = 1
        return out

    def share(self, blocks) -> None:
        """Add one reference to each block (a prefix shared by another sequence)."""
        for b in blocks:
            if self.refcount[b] <= 0:
                raise ValueError(f"sharing block {b}, which is not allocated")
            self.refcount[b] += 1

    def free(self, blocks) -> list[int]:
        """Drop one reference per block; returns the blocks that became free."""
        released = []
        for b in blocks:
            b = int(b)
            if b == self.reserved:
                raise ValueError("block 0 is reserved and never owned")
            if self.refcount[b] <= 0:
                raise ValueError(f"double free of block {b}")
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self._free.append(b)
                released.append(b)
        return released

    def check(self) -> None:
        """Conservation: every usable block is either free or owned, never both."""
        free = set(self._free)
        if len(free) != len(self._free):
            raise AssertionError("a block is on the free list twice")
        owned = set(int(b) for b in self.owned())
        if free & owned:
            raise AssertionError("a block is both free and owned")
        usable = self.num_blocks - (1 if self.reserved is not None else 0)
        if len(free) + len(owned) != usable:
            raise AssertionError("blocks leaked: free + owned != usable")
        if self.reserved is not None and (self.reserved in free or self.refcount[0] != 0):
            raise AssertionError("block 0 escaped the reservation")
