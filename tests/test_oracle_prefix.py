"""Pins for the oracle's prefix cache and copy-on-write (oracle/prefix_cache.py).

Each scenario is a statement of the pages turned into a check:
* "Text Generation Inference: Hugging Face's production-grade LLM inference
  server", "Under the Hood: PagedAttention": same system prompt -> the second
  table starts with the first one's blocks; divergent generation -> the
  written block is copied and only the writer's table changes.
* pyshine "text-generation-inference", "The radix prefix cache": block 0
  reserved; references taken before eviction; least recently used
  unreferenced prefixes evicted when the free list is empty; double-cached
  blocks back to the free list; partial overlaps split the tree.
* the same page, "Inside the batching task": a fully cached prompt gives one
  token back.
Beyond these, seeded traces check the pool's invariants and a token-content
model: every live sequence reads its own tokens through its table, every
cache hit holds the prompt's tokens. Planted mistakes (in subclasses of the
oracle, on the CPU) must fail those checks.
"""

import numpy as np
import pytest

from oracle import prefix_cache as pc
from tests.prefix_trace import PoolContent, TraceRunner

BS = 4


def toks(n, start=0):
    return list(range(start, start + n))


def test_block_zero_is_never_handed_out():
    m = pc.PrefixCacheModel(num_blocks=6, block_size=BS)
    sid, cached = m.admit(toks(5 * BS))          # exactly the 5 usable blocks
    assert cached == 0
    assert sorted(m.table(sid)) == [1, 2, 3, 4, 5]
    with pytest.raises(pc.CapacityError):
        m.admit(toks(1, 999))
    m.check()


def test_same_system_prompt_shares_the_prefix_blocks():
    m = pc.PrefixCacheModel(32, BS)
    system = toks(3 * BS + 2)                    # 3 full blocks + 2 tokens
    a, cached_a = m.admit(system + [100, 101])
    assert cached_a == 0
    m.write_slots(a, 0, len(system) + 2)
    m.release(a, system + [100, 101])
    b, cached_b = m.admit(system + [200, 201, 202])
    table_b = m.table(b)
    # the 4th block mixes the prompt's tail with A's own tokens: not shared
    assert cached_b == 3 * BS
    assert m.free.isdisjoint(table_b)
    a2, _ = m.admit(system + [100, 101])         # A's whole first 4 blocks are cached now
    table_a = m.table(a2)
    assert table_b[:3] == table_a[:3]
    assert table_b[3] != table_a[3]
    m.check()


def test_divergent_generation_copies_the_shared_block():
    m = pc.PrefixCacheModel(16, BS)
    parent, _ = m.admit(toks(BS + 2))            # block 2 of the table half full
    m.write_slots(parent, 0, BS + 2)
    child = m.fork(parent)
    assert m.table(child) == m.table(parent)
    before = m.table(parent)
    slots, copies = m.write_slots(parent, BS + 2, BS + 3)
    assert copies == [(before[1], m.table(parent)[1])]
    assert m.table(parent)[0] == before[0]       # untouched block stays shared
    assert m.table(child) == before              # the reader's table is unchanged
    assert slots == [m.table(parent)[1] * BS + 2]
    slots, copies = m.write_slots(child, BS + 2, BS + 3)
    assert copies == []                          # child now owns the original alone
    m.check()


def test_fully_cached_prompt_gives_one_token_back():
    m = pc.PrefixCacheModel(16, BS)
    p = toks(2 * BS)
    a, _ = m.admit(p)
    m.write_slots(a, 0, len(p))
    m.release(a, p)
    b, cached = m.admit(p)
    assert cached == len(p) - 1
    cached_last = m.table(b)[1]
    slots, copies = m.write_slots(b, len(p) - 1, len(p))
    assert copies and copies[0][0] == cached_last   # the cached block is not written
    assert m.table(b)[1] != cached_last
    assert m.cache[tuple(p)] == cached_last
    m.check()


def test_references_are_taken_before_eviction():
    m = pc.PrefixCacheModel(5, BS)               # 4 usable blocks
    p = toks(2 * BS)
    a, _ = m.admit(p)
    m.write_slots(a, 0, len(p))
    m.release(a, p)                              # 2 cached, unreferenced; 2 free
    b, cached = m.admit(p + toks(2 * BS, 500))   # matches 2, needs 2 more: fits exactly
    assert cached == 2 * BS
    m.check()
    m2 = pc.PrefixCacheModel(5, BS)
    a, _ = m2.admit(p)
    m2.write_slots(a, 0, len(p))
    m2.release(a, p)
    snap = (set(m2.free), dict(m2.cache), list(m2.ref))
    with pytest.raises(pc.CapacityError):        # needs 3 fresh blocks; only the match could give them
        m2.admit(p + toks(3 * BS, 500))
    assert (set(m2.free), dict(m2.cache), list(m2.ref)) == snap
    m2.check()


def test_least_recently_used_prefix_goes_first():
    m = pc.PrefixCacheModel(7, BS)               # 6 usable blocks
    prompts = [toks(2 * BS, 100 * k) for k in range(3)]
    for p in prompts:                            # three cached 2-block prefixes, ticks in order
        s, _ = m.admit(p)
        m.write_slots(s, 0, len(p))
        m.release(s, p)
    s, _ = m.admit(prompts[0])                   # touch the first again
    m.release(s, prompts[0])
    assert len(m.cache) == 6 and not m.free
    s, _ = m.admit(toks(2 * BS, 900))            # two fresh blocks: the oldest leaf chain goes
    keys = set(m.cache)
    assert tuple(prompts[1]) not in keys and tuple(prompts[1][:BS]) not in keys
    assert tuple(prompts[0]) in keys and tuple(prompts[2]) in keys
    m.check()


def test_double_cached_blocks_return_to_the_free_list():
    m = pc.PrefixCacheModel(16, BS)
    p = toks(2 * BS)
    a, _ = m.admit(p)
    b, _ = m.admit(p)                            # in flight together: nothing cached yet
    assert set(m.table(a)).isdisjoint(m.table(b))
    m.write_slots(a, 0, len(p))
    m.write_slots(b, 0, len(p))
    m.release(a, p)
    free_before = len(m.free)
    table_b = m.table(b)
    m.release(b, p)
    assert len(m.free) == free_before + 2
    assert set(table_b) <= m.free
    assert len(m.cache) == 2
    m.check()


def test_partial_overlap_splits_the_tree():
    m = pc.PrefixCacheModel(16, BS)
    x, y, z = toks(BS), toks(BS, 50), toks(BS, 90)
    a, _ = m.admit(x + y)
    m.write_slots(a, 0, 2 * BS)
    m.release(a, x + y)
    b, cached = m.admit(x + z)
    assert cached == BS
    m.write_slots(b, BS, 2 * BS)
    m.release(b, x + z)
    assert {tuple(x), tuple(x + y), tuple(x + z)} == set(m.cache)
    assert m.cache[tuple(x + y)] != m.cache[tuple(x + z)]
    m.check()


def test_copy_blocks_copies_whole_blocks_in_order():
    k = np.arange(5 * 2 * 3).reshape(5, 2, 3).astype(np.float64)
    v = -k
    want_k, want_v = k.copy(), v.copy()
    pc.copy_blocks(k, v, [(1, 3), (3, 4)])
    want_k[3] = want_k[1]
    want_v[3] = want_v[1]
    want_k[4] = want_k[3]
    want_v[4] = want_v[3]
    assert np.array_equal(k, want_k) and np.array_equal(v, want_v)


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_keep_every_sequence_intact(seed):
    m = pc.PrefixCacheModel(num_blocks=24, block_size=BS)
    run = TraceRunner(m, 24, BS, seed)
    hits = 0
    for _ in range(300):
        run.step(pc.CapacityError)
        m.check()
        run.verify_live()
    hits = sum(1 for e in run.log if e[0] == "admit" and e[2] > 0)
    copies = sum(len(e[5]) for e in run.log if e[0] == "write")
    assert hits > 5 and copies > 0               # the trace exercises sharing and CoW


class _NoCopyOnWrite(pc.PrefixCacheModel):
    def write_slots(self, sid, p0, p1):
        seq = self.seqs[sid]
        slots = []
        for p in range(p0, p1):
            i = p // self.block_size
            if i == len(seq["blocks"]):
                b = self._take()
                self.ref[b] += 1
                seq["blocks"].append(b)
            slots.append(seq["blocks"][i] * self.block_size + p % self.block_size)
        seq["ntok"] = max(seq["ntok"], p1)
        return slots, []


class _EvictReferenced(pc.PrefixCacheModel):
    def _evict_one(self):
        key = min(self.cache, key=lambda k: self.last_use[k])
        b = self.cache.pop(key)
        del self.key_of[b]
        del self.last_use[key]
        self.free.add(b)
        return b


class _NoTokenBack(pc.PrefixCacheModel):
    def admit(self, tokens):
        sid, cached = super().admit(tokens)
        if cached == len(tokens) - 1 and cached % self.block_size == self.block_size - 1:
            cached += 1
        return sid, cached


@pytest.mark.parametrize("bad", [_NoCopyOnWrite, _EvictReferenced])
def test_planted_mistakes_corrupt_sequences(bad):
    failed = False
    for seed in range(8):
        m = bad(num_blocks=24, block_size=BS)
        run = TraceRunner(m, 24, BS, seed)
        try:
            for _ in range(300):
                run.step(pc.CapacityError)
                run.verify_live()
        except (AssertionError, KeyError):
            failed = True
            break
    assert failed


def test_planted_mistake_no_token_given_back():
    m = _NoTokenBack(16, BS)
    p = toks(2 * BS)
    a, _ = m.admit(p)
    m.write_slots(a, 0, len(p))
    m.release(a, p)
    _, cached = m.admit(p)
    assert cached == len(p)                       # the pinned rule above catches this
