"""Seeded request traces for the prefix-cache tests, and a token-content model
of the pool that checks what the sharing must preserve.

A trace is a list of operations on an allocator (the oracle model or the
native one): admit a prompt (drawn from a few shared system prompts plus a
private tail), compute its uncached positions, decode a few tokens, fork a
sequence, release a sequence. `PoolContent` replays the slot writes and block
copies into a pool of token ids, so a test can check that every sequence
reads back exactly its own tokens through its table and that a cache hit
hands out blocks holding the prompt's tokens ("How to Speed Up LLM
Inference: KV Cache to Production Serving", section "The KV cache: the memory
problem that runs the show": identical prefixes give identical KV blocks).
"""

from __future__ import annotations

import numpy as np


class PoolContent:
    """Token id written at each slot (-1 = never written)."""

    def __init__(self, num_blocks: int, block_size: int):
        self.bs = block_size
        self.tok = np.full((num_blocks, block_size), -1, dtype=np.int64)

    def write(self, slots, tokens):
        for s, t in zip(slots, tokens):
            self.tok[s // self.bs, s % self.bs] = t

    def copy(self, copies):
        for src, dst in copies:
            self.tok[dst] = self.tok[src]

    def read(self, table, n):
        return [int(self.tok[table[p // self.bs], p % self.bs]) for p in range(n)]


class TraceRunner:
    """Drives an allocator through a seeded trace. `alloc` exposes admit,
    write_slots, fork, release, table, stats. Records every result so two
    allocators can be compared call by call."""

    def __init__(self, alloc, num_blocks, block_size, seed, n_prompts=3, vocab=50):
        self.a = alloc
        self.bs = block_size
        self.rng = np.random.default_rng(seed)
        self.content = PoolContent(num_blocks, block_size)
        self.prompts = [list(self.rng.integers(0, vocab, int(self.rng.integers(1, 4 * block_size))))
                        for _ in range(n_prompts)]
        self.vocab = vocab
        self.live = {}        # seq id -> tokens so far
        self.log = []

    def _compute(self, sid, p0, p1, toks):
        slots, copies = self.a.write_slots(sid, p0, p1)
        self.content.copy(copies)
        self.content.write(slots, toks[p0:p1])
        self.log.append(("write", sid, p0, p1, list(slots), list(copies)))

    def step(self, capacity_error):
        r = self.rng.random()
        if r < 0.35 or not self.live:
            base = self.prompts[int(self.rng.integers(0, len(self.prompts)))]
            tail = list(self.rng.integers(0, self.vocab, int(self.rng.integers(0, 2 * self.bs))))
            toks = list(base) + tail
            try:
                sid, cached = self.a.admit(toks)
            except capacity_error:
                self.log.append(("admit-full", len(toks)))
                return
            table = self.a.table(sid)
            assert self.content.read(table, cached) == toks[:cached], "cache hit with wrong tokens"
            self.log.append(("admit", sid, cached, list(table)))
            try:
                self._compute(sid, cached, len(toks), toks)
            except capacity_error:
                self.log.append(("write-full", sid))
                self.a.release(sid, toks[:cached])
                return
            self.live[sid] = toks
        elif r < 0.75:
            sid = list(self.live)[int(self.rng.integers(0, len(self.live)))]
            toks = self.live[sid]
            toks.append(int(self.rng.integers(0, self.vocab)))
            try:
                self._compute(sid, len(toks) - 1, len(toks), toks)
            except capacity_error:
                toks.pop()
                self.log.append(("decode-full", sid))
        elif r < 0.85:
            sid = list(self.live)[int(self.rng.integers(0, len(self.live)))]
            child = self.a.fork(sid)
            self.live[child] = list(self.live[sid])
            self.log.append(("fork", sid, child))
        else:
            sid = list(self.live)[int(self.rng.integers(0, len(self.live)))]
            toks = self.live.pop(sid)
            self.a.release(sid, toks)
            self.log.append(("release", sid))
        self.log.append(("stats",) + tuple(self.a.stats()))

    def verify_live(self):
        for sid, toks in self.live.items():
            assert self.content.read(self.a.table(sid), len(toks)) == toks, f"seq {sid} corrupted"
