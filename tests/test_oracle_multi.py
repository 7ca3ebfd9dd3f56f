"""Pins for the oracle's multi-token query attention (oracle.decode_multi):
one-token rows equal single-token decode, a prompt processed in chunks equals
full causal attention computed by torch SDPA (fp64, explicit mask), the last
row of a chunk equals decoding that token alone, a pure-Python triple loop
agrees on tiny inputs, and a planted top-left mask alignment is rejected."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P


def after_append(case):
    kc, vc = wl.bits(case.k_cache), wl.bits(case.v_cache)
    return pa.kv_append(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new),
                        case.slot_mapping.numpy())


def run(case, caches=None):
    kc, vc = caches if caches is not None else after_append(case)
    return oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)


def test_one_token_rows_equal_single_token_decode():
    case = wl.make_multi_case("m1", 1, [0, 3, 16, 40, 100], [1] * 5, 8, 2, 64, 16)
    kc, vc = after_append(case)
    got = run(case, (kc, vc))
    want = pa.decode(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                     case.context_lens.numpy(), case.scale)
    assert np.abs(got - want).max() < 1e-12


def _sdpa_causal(K, V, Q, scale, G):
    """torch SDPA, float64, on contiguous rows [n, H, D] with a causal mask."""
    q = torch.from_numpy(Q).permute(1, 0, 2)[None]                    # [1, Hq, n, D]
    k = torch.from_numpy(K).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    v = torch.from_numpy(V).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    n = Q.shape[0]
    mask = torch.ones(n, n, dtype=torch.bool).tril()
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("chunks", [[40], [16, 24], [1, 7, 16, 9, 7], [13, 27]])
def test_chunked_prefill_equals_full_causal_attention(chunks):
    n, hq, hkv, d, bs = sum(chunks), 8, 2, 64, 16
    full = wl.make_multi_case("pf", 3, [0], [n], hq, hkv, d, bs)
    kc, vc = after_append(full)                  # every position of the prompt in the pool
    K = pa.bf16_bits_to_f64(pa.gather_sequence(kc, full.block_tables.numpy()[0], n))
    V = pa.bf16_bits_to_f64(pa.gather_sequence(vc, full.block_tables.numpy()[0], n))
    Q = pa.bf16_bits_to_f64(wl.bits(full.q))
    want = _sdpa_causal(K, V, Q, full.scale, hq // hkv)
    a = 0
    for c in chunks:                             # chunk [a, a + c): context a + c
        q_rows = wl.bits(full.q)[a:a + c]
        got = oracle.decode_multi(q_rows, kc, vc, full.block_tables.numpy(),
                                  np.array([a + c]), np.array([0, c]), full.scale)
        assert np.abs(got - want[a:a + c]).max() < 1e-12, (chunks, a)
        a += c


def test_last_row_of_each_sequence_equals_decoding_it_alone():
    case = wl.make_multi_case("lr", 4, [5, 0, 33, 64], [4, 3, 8, 1], 8, 2, 64, 16)
    kc, vc = after_append(case)
    got = run(case, (kc, vc))
    qs = case.q_start.numpy()
    last = qs[1:] - 1
    want = pa.decode(wl.bits(case.q)[last], kc, vc, case.block_tables.numpy(),
                     case.context_lens.numpy(), case.scale)
    assert np.abs(got[last] - want).max() < 1e-12


def test_pure_python_triple_loop_on_tiny_inputs():
    case = wl.make_multi_case("bf", 5, [2, 0, 9], [3, 2, 2], 4, 2, 4, 4)
    kc, vc = after_append(case)
    got = run(case, (kc, vc))
    qs, ctx, bt = case.q_start.numpy(), case.context_lens.numpy(), case.block_tables.numpy()
    G, bs = 2, 4
    qf = pa.bf16_bits_to_f64(wl.bits(case.q))
    kf, vf = pa.bf16_bits_to_f64(kc), pa.bf16_bits_to_f64(vc)
    for b in range(3):
        n = qs[b + 1] - qs[b]
        for i in range(n):
            pos = ctx[b] - n + i
            for h in range(4):
                scores = []
                for t in range(pos + 1):
                    blk, off = bt[b][t // bs], t % bs
                    scores.append(case.scale * sum(qf[qs[b] + i, h, e] * kf[blk, off, h // G, e]
                                                   for e in range(4)))
                mx = max(scores)
                w = [math.exp(x - mx) for x in scores]
                for e in range(4):
                    acc = 0.0
                    for t in range(pos + 1):
                        blk, off = bt[b][t // bs], t % bs
                        acc += w[t] * vf[blk, off, h // G, e]
                    assert abs(acc / sum(w) - got[qs[b] + i, h, e]) < 1e-12


def test_rows_beyond_the_context_are_zero():
    case = wl.make_multi_case("z", 6, [0], [3], 4, 2, 64, 16)
    kc, vc = after_append(case)
    ctx = np.array([2])                          # 3 new rows, only 2 positions
    got = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(), ctx,
                              case.q_start.numpy(), case.scale)
    assert not got[0].any() and got[1:].any()


def test_planted_top_left_alignment_is_rejected():
    # a mask aligned at the chunk's start (query i sees positions 0..i) instead
    # of at its end differs from full causal attention for any later chunk
    n, hq, hkv, d, bs = 24, 4, 2, 64, 16
    full = wl.make_multi_case("tl", 7, [0], [n], hq, hkv, d, bs)
    kc, vc = after_append(full)
    K = pa.bf16_bits_to_f64(pa.gather_sequence(kc, full.block_tables.numpy()[0], n))
    V = pa.bf16_bits_to_f64(pa.gather_sequence(vc, full.block_tables.numpy()[0], n))
    Q = pa.bf16_bits_to_f64(wl.bits(full.q))
    want = _sdpa_causal(K, V, Q, full.scale, hq // hkv)
    a, c = 16, 8                                  # second chunk
    wrong = np.zeros((c, hq, d))
    for i in range(c):
        for h in range(hq):
            s = full.scale * (K[:i + 1, h // 2] @ Q[a + i, h])
            w = np.exp(s - s.max())
            wrong[i, h] = w @ V[:i + 1, h // 2] / w.sum()
    assert np.abs(wrong - want[a:a + c]).max() > 1e-3
