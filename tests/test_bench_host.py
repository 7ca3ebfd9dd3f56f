"""Host-side parts of bench.py: the causal (row, key) pair count behind
the chunked-prefill TFLOP/s, checked against a brute-force count of what the
oracle's multi-token attention reads (row at position p reads keys 0..p); the
source hash that keys recorded DRAM captures; and the reference arm's JSON
line."""

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


def test_reference_arm_prints_one_contract_line():
    # the reference arm times the oracle on the host: one JSON line with the
    # contract's keys, the bench's own metric, and its oracle baseline
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], cwd=root, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["ms_per_step"] > 0 and d["vs_baseline"] is None and d["scaling"] == "weak"
    assert d["data"] == "synthetic" and d["dtype"] == "f64" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] == 1
    assert cb["unit"] == "GB/s" and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_host_bookkeeping_replays_the_schedule_on_the_native_cache():
    # the continuous-batching schedule (finishes, joins, one token a step)
    # replayed through pa_prefix_*: the native cache's context lengths equal
    # the schedule's at every step (checked inside), and a time comes back
    from paged_kv_cache_45_gb300 import workloads as wl
    cb = wl.ContinuousBatching(seed=5, batch=48, iterations=12, p_finish=0.1)
    assert sum(len(s["finished"]) for s in cb.schedule) > 0
    ms = bench.host_bookkeeping_ms(cb)
    assert 0.0 < ms < 1e3


def test_host_bookkeeping_under_eviction_pressure():
    # the same schedule with the pool full of cached prefixes: shared system
    # prompts, finished sequences released into the cache, every fresh block
    # evicted from it; the lengths still equal the schedule's (checked inside)
    from paged_kv_cache_45_gb300 import workloads as wl
    cb = wl.ContinuousBatching(seed=5, batch=48, iterations=12, p_finish=0.1)
    ms, evicted = bench.host_bookkeeping_ms(cb, pressure=True)
    assert 0.0 < ms < 1e3
    assert evicted > 1.0
