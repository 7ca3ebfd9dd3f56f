"""The native prefix cache (pa_prefix_* in the C ABI) against the oracle's
plain model, call by call on seeded request traces: the same cached lengths,
block tables, slots, copy-on-write pairs and pool statistics. Host-only: no
GPU is touched.
"""

import numpy as np
import pytest

from oracle import prefix_cache as pc
from paged_kv_cache_45_gb300 import binding as b
from tests.prefix_trace import TraceRunner


@pytest.mark.parametrize("num_blocks,block_size,seed", [
    (24, 4, 0), (24, 4, 1), (24, 4, 2), (40, 1, 3), (40, 2, 4), (64, 16, 5), (12, 4, 6),
    (200, 4, 7), (200, 8, 8), (1000, 2, 9)])
def test_native_matches_the_oracle_call_by_call(num_blocks, block_size, seed):
    model = pc.PrefixCacheModel(num_blocks, block_size)
    native = b.PrefixCache(num_blocks, block_size)
    run_m = TraceRunner(model, num_blocks, block_size, seed)
    run_n = TraceRunner(native, num_blocks, block_size, seed)
    for step in range(400):
        run_m.step(pc.CapacityError)
        run_n.step(b.CapacityError)
        assert run_n.log == run_m.log, f"diverged at step {step}: {run_n.log[-2:]} vs {run_m.log[-2:]}"
        run_n.verify_live()
    assert any(e[0] == "admit" and e[2] > 0 for e in run_m.log)
    assert any(e[0] == "write" and e[5] for e in run_m.log)


@pytest.mark.parametrize("num_blocks,block_size,seed,n_prompts", [
    (48, 4, 21, 12), (96, 2, 22, 16), (160, 8, 23, 24), (64, 1, 24, 10)])
def test_native_matches_the_oracle_under_eviction_pressure(num_blocks, block_size, seed,
                                                           n_prompts):
    # many distinct system prompts in a small pool: the cache fills it and
    # most admits and writes must evict least recently used prefixes first.
    # Besides the call-by-call log, the count of blocks eviction could free
    # (kept incrementally by the native cache) equals the model's walk.
    model = pc.PrefixCacheModel(num_blocks, block_size)
    native = b.PrefixCache(num_blocks, block_size)
    evictions = []
    evict = model._evict_one

    def counting_evict():
        evictions.append(1)
        return evict()

    model._evict_one = counting_evict
    run_m = TraceRunner(model, num_blocks, block_size, seed, n_prompts=n_prompts)
    run_n = TraceRunner(native, num_blocks, block_size, seed, n_prompts=n_prompts)
    for step in range(1200):
        run_m.step(pc.CapacityError)
        run_n.step(b.CapacityError)
        assert run_n.log == run_m.log, f"diverged at step {step}: {run_n.log[-2:]} vs {run_m.log[-2:]}"
        assert native.evictable() == model._evictable(), f"evictable count at step {step}"
        run_n.verify_live()
    assert len(evictions) > 100
    assert any(e[0] == "admit-full" for e in run_m.log) or len(evictions) > 300


def test_append_tokens_equals_one_write_per_sequence():
    bs = 4
    a, c = b.PrefixCache(64, bs), pc.PrefixCacheModel(64, bs)
    seqs_a, seqs_c = [], []
    prompt = list(range(2 * bs))
    for alloc, seqs in ((a, seqs_a), (c, seqs_c)):
        s0, _ = alloc.admit(prompt)
        alloc.write_slots(s0, 0, len(prompt))
        alloc.release(s0, prompt)
        for k in range(5):
            sid, cached = alloc.admit(prompt + [100 + k])
            alloc.write_slots(sid, cached, len(prompt) + 1)
            seqs.append(sid)
        seqs.append(alloc.fork(seqs[0]))
    slots, (src, dst) = a.append_tokens(seqs_a)
    want_slots, want_copies = [], []
    for sid in seqs_c:
        n = c.seqs[sid]["ntok"]
        sl, cp = c.write_slots(sid, n, n + 1)
        want_slots += sl
        want_copies += cp
    assert list(slots) == want_slots
    assert list(zip(src.tolist(), dst.tolist())) == want_copies
    assert want_copies                          # the fork's shared block was copied
    tables, lens = a.tables(seqs_a, 8)
    for i, sid in enumerate(seqs_c):
        t = c.table(sid)
        assert tables[i, :len(t)].tolist() == t and not tables[i, len(t):].any()
        assert lens[i] == c.seqs[sid]["ntok"]


def test_capacity_error_changes_nothing():
    bs = 4
    a = b.PrefixCache(6, bs)                     # 5 usable blocks
    s, _ = a.admit(list(range(3 * bs)))
    before = (a.stats(), a.table(s))
    with pytest.raises(b.CapacityError):
        a.admit(list(range(100, 100 + 3 * bs)))
    with pytest.raises(b.CapacityError):
        a.write_slots(s, 3 * bs, 6 * bs)
    assert (a.stats(), a.table(s)) == before
    a.write_slots(s, 3 * bs, 5 * bs)            # exactly what is left
    assert a.stats()[0] == 0


def test_invalid_arguments_are_rejected():
    a = b.PrefixCache(16, 4)
    with pytest.raises(b.PagedKVError):
        a.admit([])
    s, _ = a.admit([1, 2, 3])
    for call in (lambda: a.write_slots(s, 5, 6),          # a hole after the sequence
                 lambda: a.write_slots(s + 99, 0, 1),     # unknown sequence
                 lambda: a.fork(s + 99),
                 lambda: a.release(s + 99, [1])):
        with pytest.raises(b.PagedKVError) as e:
            call()
        assert e.value.status == -1
    with pytest.raises(b.PagedKVError):
        b.PrefixCache(1, 4)
    assert b.pa_status_str(-6) == "PA_ERR_CAPACITY"


def test_block_zero_is_never_used_and_the_pool_is_conserved():
    nb, bs = 50, 2
    a = b.PrefixCache(nb, bs)
    run = TraceRunner(a, nb, bs, seed=11)
    for _ in range(500):
        run.step(b.CapacityError)
        free, cached, used = a.stats()
        assert free + cached + used >= nb - 1 >= free
        for sid in run.live:
            assert 0 not in a.table(sid)
    run.verify_live()


def test_fork_batch_and_discard_equal_their_single_calls():
    bs = 4
    a, c = b.PrefixCache(40, bs), pc.PrefixCacheModel(40, bs)
    ids_a, ids_c = [], []
    for k in range(4):
        p = list(range(10 * k, 10 * k + 6))
        ids_a.append(a.admit(p)[0])
        ids_c.append(c.admit(p)[0])
        a.write_slots(ids_a[-1], 0, 6)
        c.write_slots(ids_c[-1], 0, 6)
    kids_a = a.fork_batch(ids_a).tolist()
    kids_c = [c.fork(s) for s in ids_c]
    assert kids_a == kids_c
    slots, (src, dst) = a.append_tokens(kids_a)
    want = [c.write_slots(s, 6, 7) for s in kids_c]
    assert list(slots) == [w[0][0] for w in want]
    assert list(zip(src.tolist(), dst.tolist())) == [w[1][0] for w in want]
    a.discard(kids_a)
    for s in kids_c:
        c.release(s, [])
    assert a.stats() == c.stats()
    for sa, sc in zip(ids_a, ids_c):
        assert a.table(sa) == c.table(sc)


def test_fresh_blocks_lowest_first_across_a_large_pool():
    # most of a 2000-block pool taken, a random half of the sequences ended
    # (their blocks back on the free list in scattered order), then refilled:
    # every table equals the oracle model's, which takes the lowest free id
    rng = np.random.default_rng(11)
    nb, bs = 2000, 2
    model, native = pc.PrefixCacheModel(nb, bs), b.PrefixCache(nb, bs)
    live, uid = [], 0
    for rnd in range(3):
        while True:
            n = int(rng.integers(1, 60))
            if native.stats()[0] < -(-n // bs):
                break
            uid += 1
            toks = [uid * 1000 + i for i in range(n)]     # no shared prefixes
            sid_m, _ = model.admit(toks)
            sid_n, _ = native.admit(toks)
            assert sid_m == sid_n
            live.append(sid_n)
        for sid in live:
            assert native.table(sid) == model.table(sid)
        assert native.stats() == model.stats()
        ended = [s for s in live if rng.random() < 0.5]
        for sid in ended:
            model.release(sid, [])
        native.discard(ended)
        live = [s for s in live if s not in ended]
        assert native.stats() == model.stats()
