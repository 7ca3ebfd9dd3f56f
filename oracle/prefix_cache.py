"""Plain model of the paged block pool with a prefix cache and copy-on-write.

TEST INFRASTRUCTURE ONLY. Nothing in the product imports this module; the
tests compare the library's native allocator and its block-copy kernel with
it, and it is pinned by tests/test_oracle_prefix.py to the behaviour the pages
describe.

What it follows:

* "Text Generation Inference: Hugging Face's production-grade LLM inference
  server", section "Under the Hood: PagedAttention" (prefix sharing): requests
  with the same system prompt point their block tables at the same physical
  blocks; a write into a shared block first copies it to a fresh block and
  repoints the writer's table (copy-on-write).
* pyshine "text-generation-inference", section "The radix prefix cache":
  block 0 is reserved; a free list plus a prefix tree keyed by the token ids
  at block granularity; allocation matches the request's tokens, takes a
  reference on the matched blocks before anything may be evicted, then takes
  fresh blocks for the suffix, evicting the least recently used unreferenced
  prefixes when the free list is empty; on release, the request's computed
  prefix goes into the tree and blocks whose prefix another request cached in
  the meantime go back to the free list.
* the same page, section "Inside the batching task": when the cache holds the
  whole prompt, one token is given back so that at least one position is
  computed fresh.
* "How to Speed Up LLM Inference: KV Cache to Production Serving", section
  "The KV cache: the memory problem that runs the show" (items 1 and 2):
  blocks shared copy-on-write between sequences; identical prefixes give
  identical KV blocks, which is what makes reuse sound.

Readings where the pages leave a step open (each one is a rule below):

* Only full blocks are cached; a cached block is keyed by the whole token
  prefix it ends (so equal keys mean equal K/V content).
* The tree is modelled by that dict of prefixes (a compressed tree holds the
  same set of keys); a block is a leaf when no cached key extends its key by
  one block.
* Eviction removes one block at a time: the leaf with the oldest use tick
  among leaves no sequence references. Every public call advances one tick;
  matching, inserting and touching on release stamp the keys on the request's
  path with it.
* Fresh blocks are taken lowest id first.
* A write into a block that is cached or referenced by another sequence is a
  copy-on-write of the whole block.
* A call that needs more fresh blocks than the free blocks plus the blocks
  eviction could free at its start (cached, unreferenced, nothing referenced
  cached below them) fails before changing anything.

Written as plain data structures and loops, favouring obviousness over speed.
"""

from __future__ import annotations

import numpy as np


class CapacityError(RuntimeError):
    """No free block and nothing evictable."""


class PrefixCacheModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 2 or block_size < 1:
            raise ValueError("need at least one usable block")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = set(range(1, num_blocks))      # block 0 is reserved
        self.ref = [0] * num_blocks                 # live sequences using the block
        self.cache = {}                             # prefix tuple -> block id
        self.key_of = {}                            # block id -> prefix tuple
        self.last_use = {}                          # prefix tuple -> tick
        self.tick = 0
        self.seqs = {}                              # seq id -> {"blocks": [...], "ntok": int}
        self.next_seq = 1

    # ------------------------------------------------------------ internals
    def _is_leaf(self, key) -> bool:
        n = len(key) + self.block_size
        for other in self.cache:
            if len(other) == n and other[:len(key)] == key:
                return False
        return True

    def _evict_one(self) -> int:
        best = None
        for key, b in self.cache.items():
            if self.ref[b] == 0 and self._is_leaf(key):
                cand = (self.last_use[key], b)
                if best is None or cand < best[0]:
                    best = (cand, key, b)
        if best is None:
            raise CapacityError("pool exhausted")
        _, key, b = best
        del self.cache[key]
        del self.key_of[b]
        del self.last_use[key]
        self.free.add(b)
        return b

    def _evictable(self) -> int:
        count = 0
        for key, b in self.cache.items():
            if self.ref[b] != 0:
                continue
            below = [b2 for k2, b2 in self.cache.items()
                     if len(k2) > len(key) and k2[:len(key)] == key]
            if all(self.ref[b2] == 0 for b2 in below):
                count += 1
        return count

    def _reserve(self, needed: int):
        if needed > len(self.free) + self._evictable():
            raise CapacityError("pool exhausted")

    def _take(self) -> int:
        if not self.free:
            self._evict_one()
        b = min(self.free)
        self.free.remove(b)
        return b

    def _drop_ref(self, b: int):
        self.ref[b] -= 1
        if self.ref[b] == 0 and b not in self.key_of:
            self.free.add(b)

    # ------------------------------------------------------------- the API
    def admit(self, tokens):
        """Match `tokens` against the cache and give the new sequence blocks
        for positions [0, len(tokens)). Returns (seq id, cached tokens): the
        K/V of positions < cached tokens are already in the sequence's
        blocks."""
        tokens = tuple(int(t) for t in tokens)
        n = len(tokens)
        if n < 1:
            raise ValueError("empty prompt")
        self.tick += 1
        bs = self.block_size
        matched = []
        while (len(matched) + 1) * bs <= n:
            key = tokens[:(len(matched) + 1) * bs]
            if key not in self.cache:
                break
            matched.append(self.cache[key])
        for b in matched:                        # references first: no eviction can take them
            self.ref[b] += 1
        try:
            self._reserve(-(-n // bs) - len(matched))
        except CapacityError:
            for b in matched:
                self.ref[b] -= 1
            raise
        for i in range(len(matched)):
            self.last_use[tokens[:(i + 1) * bs]] = self.tick
        blocks = list(matched)
        while len(blocks) * bs < n:
            b = self._take()
            self.ref[b] += 1
            blocks.append(b)
        cached = len(matched) * bs
        if cached == n:
            cached = n - 1                        # one position is always computed
        sid = self.next_seq
        self.next_seq += 1
        self.seqs[sid] = {"blocks": blocks, "ntok": n}
        return sid, cached

    def write_slots(self, sid: int, p0: int, p1: int):
        """Slots for writing positions [p0, p1) of a sequence, growing it as
        needed. A write into a block that is cached or shared first copies the
        block. Returns (slots, copies) with copies a list of (src, dst)."""
        seq = self.seqs[sid]
        if not 0 <= p0 <= seq["ntok"] or p1 < p0:
            raise ValueError("positions must continue the sequence")
        self.tick += 1
        bs = self.block_size
        needed = 0
        for i in range(p0 // bs, (p1 - 1) // bs + 1 if p1 > p0 else p0 // bs):
            if i >= len(seq["blocks"]):
                needed += 1
            else:
                b = seq["blocks"][i]
                if self.ref[b] > 1 or b in self.key_of:
                    needed += 1
        self._reserve(needed)
        slots, copies = [], []
        for p in range(p0, p1):
            i = p // bs
            if i == len(seq["blocks"]):
                b = self._take()
                self.ref[b] += 1
                seq["blocks"].append(b)
            else:
                old = seq["blocks"][i]
                if self.ref[old] > 1 or old in self.key_of:
                    new = self._take()
                    self.ref[new] += 1
                    copies.append((old, new))
                    seq["blocks"][i] = new
                    self._drop_ref(old)
            slots.append(seq["blocks"][i] * bs + p % bs)
        seq["ntok"] = max(seq["ntok"], p1)
        return slots, copies

    def fork(self, sid: int) -> int:
        """A new sequence sharing every block of `sid` (parallel sampling)."""
        seq = self.seqs[sid]
        self.tick += 1
        for b in seq["blocks"]:
            self.ref[b] += 1
        child = self.next_seq
        self.next_seq += 1
        self.seqs[child] = {"blocks": list(seq["blocks"]), "ntok": seq["ntok"]}
        return child

    def release(self, sid: int, tokens):
        """The sequence ends with K/V computed for `tokens` (positions
        [0, len(tokens))). Its full blocks enter the cache unless their prefix
        is cached already; then every reference it holds is dropped."""
        seq = self.seqs.pop(sid)
        self.tick += 1
        tokens = tuple(int(t) for t in tokens)
        bs = self.block_size
        nfull = min(len(tokens), seq["ntok"]) // bs
        for i in range(nfull):
            key = tokens[:(i + 1) * bs]
            b = seq["blocks"][i]
            if key not in self.cache:
                if b in self.key_of:     # the block holds another prefix: stop here
                    break
                self.cache[key] = b
                self.key_of[b] = key
            self.last_use[key] = self.tick
        for b in seq["blocks"]:
            self._drop_ref(b)

    def table(self, sid: int):
        return list(self.seqs[sid]["blocks"])

    def stats(self):
        """(free blocks, cached blocks, blocks referenced by sequences)."""
        return len(self.free), len(self.cache), sum(1 for r in self.ref if r > 0)

    def check(self):
        """The pool's invariants; raises AssertionError when one fails."""
        assert 0 not in self.free and 0 not in self.key_of and self.ref[0] == 0
        counted = [0] * self.num_blocks
        for s in self.seqs.values():
            for b in s["blocks"]:
                counted[b] += 1
        assert counted == self.ref, "refcounts"
        for b in self.free:
            assert self.ref[b] == 0 and b not in self.key_of, "free block in use"
        live = {b for b in range(1, self.num_blocks) if self.ref[b] > 0 or b in self.key_of}
        assert len(self.free) + len(live) == self.num_blocks - 1, "conservation"
        assert all(self.cache[k] == b for b, k in self.key_of.items())
        for key in self.cache:                     # a cached key's parent is cached
            if len(key) > self.block_size:
                assert key[:-self.block_size] in self.cache, "orphan"


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, copies) -> None:
    """Copy-on-write on the pools ([NB, bs, ...] arrays): block dst becomes a
    byte copy of block src, for each pair in order."""
    for src, dst in copies:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
