"""Host-side arithmetic of bench.py: the causal (row, key) pair count behind
the chunked-prefill TFLOP/s, checked against a brute-force count of what the
oracle's multi-token attention reads (row at position p reads keys 0..p)."""

import numpy as np

import bench


def brute(q_start, ctx):
    total = 0
    for b in range(len(ctx)):
        n = q_start[b + 1] - q_start[b]
        for i in range(n):
            pos = ctx[b] - n + i
            total += max(pos + 1, 0)
    return total


def test_attended_pairs_matches_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(200):
        B = int(rng.integers(1, 6))
        n = rng.integers(0, 40, B)
        ctx = rng.integers(0, 60, B)          # some contexts shorter than the chunk
        qs = np.concatenate([[0], np.cumsum(n)])
        assert bench.attended_pairs(qs, ctx) == brute(qs, ctx)


def test_prefill_step_flops():
    # 8 sequences x 2048 new tokens after 6144 cached: rows see 6145..8192 keys
    qs = np.arange(9) * 2048
    ctx = np.full(8, 8192)
    pairs = bench.attended_pairs(qs, ctx)
    assert pairs == 8 * sum(range(6145, 8193))
    assert 4 * 128 * 64 * pairs == 3848559132672   # the bench line's FLOPs per launch


def test_source_hash_ignores_comments_only():
    a = "int f(int x) {  // doubles\n  /* the rest\n     of it */ return 2 * x;\n}\n"
    b = "int f(int x) {\n\n  return 2 * x;   \n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench.code_of(a) == bench.code_of(b)
    assert bench.code_of(a) != bench.code_of(c)
