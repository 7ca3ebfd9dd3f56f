"""Host logic: the block allocator's invariants and the seeded generators."""

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from paged_kv_cache_45_gb300.allocator import BlockAllocator, PoolExhausted


def test_allocator_never_hands_out_block_0_and_conserves():
    a = BlockAllocator(9, order=[5, 3, 1, 8, 2, 7, 4, 6])
    got = a.allocate(8)
    assert got == [5, 3, 1, 8, 2, 7, 4, 6] and 0 not in got
    with pytest.raises(PoolExhausted):
        a.allocate(1)
    a.share([3, 1])
    assert a.free([3, 1, 5]) == [5]          # shared blocks survive one release
    assert a.free([3, 1]) == [3, 1]
    with pytest.raises(ValueError):
        a.free([3])                           # double free
    with pytest.raises(ValueError):
        a.free([0])                           # reserved
    a.check()
    assert a.num_free == 3


def test_allocator_rejects_bad_order():
    with pytest.raises(ValueError):
        BlockAllocator(4, order=[1, 2, 2])


def test_continuous_batching_schedule_invariants():
    cb = wl.ContinuousBatching(seed=0)          # full 70B-shape schedule, no tensors
    assert cb.B == 256 and cb.Hq == 64 and cb.Hkv == 8 and cb.D == 128
    finished = 0
    prev = None
    for it, s in enumerate(cb.schedule):
        lens = s["lens"].numpy()
        tabs = s["tables"].numpy()
        assert lens.min() >= 1 and lens.max() <= cb.max_blocks * cb.bs
        owned = []
        for b in range(cb.B):
            n = -(-int(lens[b]) // cb.bs)
            owned += tabs[b, :n].tolist()
            assert 0 not in tabs[b, :n]
            assert s["slots"][b] // cb.bs == tabs[b, (lens[b] - 1) // cb.bs]
            assert s["slots"][b] % cb.bs == (lens[b] - 1) % cb.bs
        assert len(owned) == len(set(owned)), "a block is owned twice"
        if prev is not None:
            grown = [b for b in range(cb.B) if b not in s["finished"]]
            assert np.all(lens[grown] == prev[grown] + 1)
        finished += len(s["finished"])
        prev = lens
    cb.alloc.check()
    assert finished > 0                       # the churn actually happened
    assert cb.alloc.num_free > 0              # the pool never ran dry


def test_continuous_batching_steps_are_reproducible_alone():
    cb1 = wl.ContinuousBatching(seed=3, batch=16, ctx_hi=512, prompt_hi=256, iterations=6,
                                p_finish=0.2)
    cb2 = wl.ContinuousBatching(seed=3, batch=16, ctx_hi=512, prompt_hi=256, iterations=6,
                                p_finish=0.2)
    a, b = cb1.step(4), cb2.step(4)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.fill_slots, b.fill_slots)
    assert torch.equal(a.block_tables, b.block_tables)


def test_continuous_batching_fills_match_joiners():
    cb = wl.ContinuousBatching(seed=4, batch=16, ctx_hi=512, prompt_hi=256, iterations=8,
                               p_finish=0.25)
    for it in range(cb.iterations):
        st = cb.step(it)
        joins = cb.schedule[it]["joins"]
        assert st.fill_slots.numel() == sum(p for _, p in joins) == st.fill_k.shape[0]
        for b, plen in joins:
            assert int(st.context_lens[b]) == plen + 1


def test_generators_are_deterministic_and_seed_dependent():
    a, b, c = wl.tiny_case(0), wl.tiny_case(0), wl.tiny_case(1)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert not torch.equal(a.q.view(torch.int16), c.q.view(torch.int16))


def test_tiny_case_shape():
    c = wl.tiny_case(0)
    assert c.context_lens.tolist() == [2, 8, 17, 34]
    assert c.num_blocks == 16 and c.block_size == 16 and c.head_dim == 64
    assert [len(b) for b in c.seq_blocks] == [1, 1, 2, 3]
    # slot of the appended token: 16 -> 17 opens a fresh block at offset 0
    assert int(c.slot_mapping[2]) % 16 == 0
    assert 0 not in np.concatenate(c.seq_blocks)


def test_unowned_slots_are_nan_poisoned():
    c = wl.make_case("p", 0, [5, 20], 2, 1, 16, 16)
    kb = wl.bits(c.k_cache)
    nan_rows = (kb == wl.BF16_NAN_BITS).all(axis=(2, 3))
    owned_rows = np.zeros_like(nan_rows)
    for b, blocks in enumerate(c.seq_blocks):
        rows = wl.token_rows(blocks, int(c.meta["ctx_before"][b]), 16)
        owned_rows.reshape(-1)[rows] = True
    assert np.array_equal(~nan_rows, owned_rows)
    assert nan_rows[0].all()                  # block 0


def test_long_context_outliers_scaled_by_8():
    c = wl.make_case("l", 1, [1000], 2, 1, 16, 16, append=False, k_outlier_frac=0.01)
    K = pa.bf16_bits_to_f64(pa.gather_sequence(wl.bits(c.k_cache), c.block_tables[0].numpy(), 1000))
    big = np.abs(K).max(axis=(1, 2))
    assert (big > 8).sum() >= 5               # ~10 rows x8 leave N(0,1) range
