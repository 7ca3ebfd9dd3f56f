"""Pins for the CPU oracle: each test ties it to something other than itself.

Facts used: the pages' printed KV sizes (golden fixture), closed forms of
softmax attention (one token, two tokens, identical keys, empty context), the
page-table property that physical block ids are only names (permutation and
block-size invariance, shared-vs-copied prefix), the streaming-softmax
recurrence and the split/merge algebra (exact reorderings of the same sum),
an independent library routine (torch's scaled_dot_product_attention, fp64,
CPU) and brute-force scalar loops in the pages' own loop structure.

``test_pins_catch_planted_mistakes`` plants plausible mistakes in copies of
the oracle and checks that these pins reject every one.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes_per_token.txt")
UNITS = {"B": 1, "KiB": 1024, "MiB": 1024 ** 2, "GiB": 1024 ** 3}


def f2b(x) -> np.ndarray:
    """Exactly representable floats -> bfloat16 bit patterns (uint16)."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bfloat16"
    return (u >> 16).astype(np.uint16)


def case_bits(c):
    return (wl.bits(c.q), wl.bits(c.k_cache), wl.bits(c.v_cache),
            c.block_tables.numpy(), c.context_lens.numpy())


def appended(c):
    """Oracle caches after the case's append step (if any)."""
    kc, vc = wl.bits(c.k_cache), wl.bits(c.v_cache)
    if c.k_new is None:
        return kc, vc
    return pa.kv_append(kc, vc, wl.bits(c.k_new), wl.bits(c.v_new), c.slot_mapping.numpy())


def small_case(seed=0, lens=(1, 5, 16, 17, 40, 3), hq=8, hkv=2, d=64, bs=16, **kw):
    return wl.make_case("small", seed, list(lens), hq, hkv, d, bs, **kw)


def run_decode(c, fn=pa.decode, **kw):
    kc, vc = appended(c)
    return fn(wl.bits(c.q), kc, vc, c.block_tables.numpy(), c.context_lens.numpy(),
              c.scale, **kw)


# ---------------------------------------------------------------------------
# 1. the bytes-per-token formula against the pages' printed numbers
# ---------------------------------------------------------------------------

def golden_rows():
    rows = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lab, L, H, D, b, tok, seqs, exp, unit = line.split()
            rows.append((lab, int(L), int(H), int(D), int(b), int(tok), int(seqs),
                         float(exp) * UNITS[unit]))
    return rows


@pytest.mark.parametrize("row", golden_rows(), ids=lambda r: r[0])
def test_kv_bytes_formula_matches_printed_figures(row):
    lab, L, H, D, b, tok, seqs, expected = row
    got = oracle.kv_bytes_per_token(L, H, D, b) * tok * seqs
    assert got == expected, (lab, got, expected)


def test_golden_fixture_is_complete():
    assert len(golden_rows()) == 22


def test_deepseek_row_does_not_follow_the_formula():
    # The table's DeepSeek V3 row prints 1,048,576 B/token for 67 layers x 16
    # KV heads x 128 x BF16; the formula gives 548,864. Kept out of the pins.
    assert oracle.kv_bytes_per_token(67, 16, 128, 2) == 548_864 != 1_048_576


# ---------------------------------------------------------------------------
# 2. closed forms
# ---------------------------------------------------------------------------

def _one_seq_pool(K, V, bs=4, nb=8, perm_seed=0):
    """Place logical rows K, V ([ctx, 1, D] uint16) into a NaN pool."""
    ctx, d = K.shape[0], K.shape[-1]
    rng = np.random.default_rng(perm_seed)
    nblk = -(-ctx // bs)
    phys = (1 + rng.permutation(nb - 1))[:nblk]
    kc = np.full((nb, bs, 1, d), wl.BF16_NAN_BITS, np.uint16)
    vc = kc.copy()
    for t in range(ctx):
        kc[phys[t // bs], t % bs] = K[t]
        vc[phys[t // bs], t % bs] = V[t]
    table = np.zeros((1, nb), np.int32)
    table[0, :nblk] = phys
    return kc, vc, table


def test_context_of_one_returns_v_exactly():
    rng = np.random.default_rng(1)
    d = 64
    q = f2b(np.round(rng.normal(size=(1, 3, d)) * 8) / 8)        # 3 q heads on 1 KV head
    K = f2b(np.round(rng.normal(size=(1, 1, d)) * 8) / 8)
    V = f2b(np.round(rng.normal(size=(1, 1, d)) * 8) / 8)
    kc, vc, tab = _one_seq_pool(K, V)
    out = oracle.decode(q, kc, vc, tab, np.array([1]), 0.125)
    for h in range(3):
        np.testing.assert_array_equal(out[0, h], pa.bf16_bits_to_f64(V[0, 0]))


def test_two_tokens_closed_form():
    # out = (V0 + e^D V1) / (1 + e^D), D = scale * q.(k1 - k0)
    d = 8
    q = np.zeros((1, 1, d), np.float32); q[0, 0, :3] = [1.0, -2.0, 0.5]
    k = np.zeros((2, 1, d), np.float32); k[0, 0, :3] = [0.5, 1.0, 2.0]; k[1, 0, :3] = [3.0, -1.0, -4.0]
    v = np.zeros((2, 1, d), np.float32); v[0, 0, :] = np.arange(d); v[1, 0, :] = -2.0 * np.arange(d) + 1
    scale = 0.25
    kc, vc, tab = _one_seq_pool(f2b(k), f2b(v), bs=1, nb=4)
    out = oracle.decode(f2b(q), kc, vc, tab, np.array([2]), scale)
    delta = scale * float(q[0, 0] @ (k[1, 0] - k[0, 0]))
    e = math.exp(delta)
    v64 = v.astype(np.float64)
    expected = (v64[0, 0] + e * v64[1, 0]) / (1.0 + e)
    np.testing.assert_allclose(out[0, 0], expected, rtol=1e-13, atol=1e-13)


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(2)
    ctx, d = 37, 64
    q = f2b(np.round(rng.normal(size=(1, 2, d)) * 4) / 4)
    krow = np.round(rng.normal(size=(1, 1, d)) * 4) / 4
    K = f2b(np.repeat(krow, ctx, axis=0))
    V = f2b(np.round(rng.normal(size=(ctx, 1, d)) * 4) / 4)
    kc, vc, tab = _one_seq_pool(K, V, bs=16, nb=8)
    out = oracle.decode(q, kc, vc, tab, np.array([ctx]), 0.125)
    mean = pa.bf16_bits_to_f64(V[:, 0]).mean(axis=0)
    for h in range(2):
        np.testing.assert_allclose(out[0, h], mean, rtol=0, atol=1e-12)


def test_empty_context_gives_zeros():
    c = small_case(lens=(0, 4), append=False)
    out = run_decode(c)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out))


# ---------------------------------------------------------------------------
# 3. page-table invariances (block ids are names only)
# ---------------------------------------------------------------------------

def test_permutation_of_physical_blocks_is_invisible():
    c = small_case(seed=3)
    q, kc, vc, bt, cl = case_bits(c)
    kc, vc = appended(c)
    base = pa.decode(q, kc, vc, bt, cl, c.scale)
    rng = np.random.default_rng(5)
    pi = np.concatenate([[0], 1 + rng.permutation(kc.shape[0] - 1)])   # pi[old] = new
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = pi[bt].astype(np.int32)
    np.testing.assert_array_equal(pa.decode(q, kc2, vc2, bt2, cl, c.scale), base)


def _relayout(kc, bt, cl, new_bs, nb_new, seed):
    """Same logical rows, re-placed into a pool of another block size."""
    rng = np.random.default_rng(seed)
    H, D = kc.shape[2], kc.shape[3]
    B = len(cl)
    need = [-(-int(c) // new_bs) for c in cl]
    order = 1 + rng.permutation(nb_new - 1)
    pool = np.full((nb_new, new_bs, H, D), wl.BF16_NAN_BITS, np.uint16)
    tab = np.zeros((B, max(max(need), 1)), np.int32)
    k = 0
    for b in range(B):
        rows = pa.gather_sequence(kc, bt[b], int(cl[b]))
        for j in range(need[b]):
            tab[b, j] = order[k]; k += 1
        for t in range(int(cl[b])):
            pool[tab[b, t // new_bs], t % new_bs] = rows[t]
    return pool, tab


def test_block_size_1_and_16_give_identical_results():
    c = small_case(seed=4, bs=16)
    q, _, _, bt, cl = case_bits(c)
    kc, vc = appended(c)
    base = pa.decode(q, kc, vc, bt, cl, c.scale)
    nb1 = int(cl.sum()) + 10
    kc1, tab1 = _relayout(kc, bt, cl, 1, nb1, seed=9)
    vc1, tab1v = _relayout(vc, bt, cl, 1, nb1, seed=9)
    np.testing.assert_array_equal(tab1, tab1v)
    np.testing.assert_array_equal(pa.decode(q, kc1, vc1, tab1, cl, c.scale), base)


def test_shared_prefix_equals_copied_prefix():
    c = wl.make_case("pfx", 6, [48 + 5, 48 + 20, 48 + 33], 4, 1, 64, 16, shared_prefix=48)
    q, _, _, bt, cl = case_bits(c)
    kc, vc = appended(c)
    assert (bt[:, :3] == bt[0, :3]).all()       # same physical prefix blocks everywhere
    base = pa.decode(q, kc, vc, bt, cl, c.scale)
    # copy the prefix into private blocks for sequences 1 and 2
    nb = kc.shape[0]
    kc2 = np.concatenate([kc, np.repeat(kc[bt[0, :3]], 2, axis=0)])
    vc2 = np.concatenate([vc, np.repeat(vc[bt[0, :3]], 2, axis=0)])
    kc2[nb:nb + 3] = kc[bt[0, :3]]; kc2[nb + 3:] = kc[bt[0, :3]]
    vc2[nb:nb + 3] = vc[bt[0, :3]]; vc2[nb + 3:] = vc[bt[0, :3]]
    bt2 = bt.copy()
    bt2[1, :3] = np.arange(nb, nb + 3)
    bt2[2, :3] = np.arange(nb + 3, nb + 6)
    np.testing.assert_array_equal(pa.decode(q, kc2, vc2, bt2, cl, c.scale), base)


# ---------------------------------------------------------------------------
# 4. exact reorderings: streaming softmax, splits + log-sum-exp merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("tile", [1, 7, 16, 64])
def test_online_recurrence_equals_two_pass(tile):
    c = small_case(seed=7, lens=(1, 15, 16, 31, 100, 250))
    np.testing.assert_allclose(run_decode(c, pa.decode_online, tile=tile), run_decode(c),
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("split", [16, 32, 64, 4096])
def test_split_then_merge_equals_unsplit(split):
    c = small_case(seed=8, lens=(0, 1, 15, 16, 31, 100, 250))
    kc, vc = appended(c)
    cl = c.context_lens.numpy()
    S = max(1, -(-int(cl.max()) // split))
    po, pl = pa.decode_split_partials(wl.bits(c.q), kc, vc, c.block_tables.numpy(), cl,
                                      c.scale, split, S + 2)        # 2 always-empty splits
    assert np.all(np.isneginf(pl[:, :, S:]))
    merged = pa.lse_merge(po, pl)
    np.testing.assert_allclose(merged, run_decode(c), rtol=0, atol=1e-12)


def test_split_lse_is_log_sum_exp_of_scores():
    c = small_case(seed=10, lens=(40,), hq=2, hkv=1)
    kc, vc = appended(c)
    cl = c.context_lens.numpy()
    po, pl = pa.decode_split_partials(wl.bits(c.q), kc, vc, c.block_tables.numpy(), cl,
                                      c.scale, 16, 3)
    K = pa.bf16_bits_to_f64(pa.gather_sequence(kc, c.block_tables.numpy()[0], int(cl[0])))
    qf = pa.bf16_bits_to_f64(wl.bits(c.q))
    for h in range(2):
        s = c.scale * (K[:, 0, :] @ qf[0, h])
        for sp in range(3):
            seg = s[16 * sp:16 * (sp + 1)]
            assert abs(pl[0, h, sp] - math.log(sum(math.exp(x) for x in seg))) < 1e-12


# ---------------------------------------------------------------------------
# 5. an independent library routine and brute force
# ---------------------------------------------------------------------------

def sdpa_reference(c):
    """torch.nn.functional.scaled_dot_product_attention, fp64 CPU, with K/V rows
    gathered by tensor indexing and repeated per query head of the group."""
    kc, vc = appended(c)
    q = torch.from_numpy(pa.bf16_bits_to_f64(wl.bits(c.q)))
    kc_t = torch.from_numpy(pa.bf16_bits_to_f64(kc))
    vc_t = torch.from_numpy(pa.bf16_bits_to_f64(vc))
    G = c.num_q_heads // c.num_kv_heads
    outs = []
    for b in range(c.batch):
        ctx = int(c.context_lens[b])
        if ctx == 0:
            outs.append(torch.zeros(c.num_q_heads, c.head_dim, dtype=torch.float64))
            continue
        t = torch.arange(ctx)
        blk = c.block_tables[b].long()[t // c.block_size]
        K = kc_t[blk, t % c.block_size]                     # [ctx, Hkv, D]
        V = vc_t[blk, t % c.block_size]
        K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, ctx, D]
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].unsqueeze(1), K, V, scale=c.scale)          # [Hq, 1, D]
        outs.append(o[:, 0])
    return torch.stack(outs).numpy()


@pytest.mark.parametrize("seed,hq,hkv,d,bs", [(11, 8, 2, 64, 16), (12, 4, 4, 32, 8),
                                              (13, 8, 1, 128, 32), (14, 6, 3, 16, 1)])
def test_matches_torch_sdpa(seed, hq, hkv, d, bs):
    c = small_case(seed=seed, lens=(0, 1, 9, 16, 47, 130), hq=hq, hkv=hkv, d=d, bs=bs)
    np.testing.assert_allclose(run_decode(c), sdpa_reference(c), rtol=0, atol=1e-12)


@pytest.mark.parametrize("d,bs", [(4, 1), (4, 8), (64, 16), (64, 32)])
def test_matches_scalar_loops_in_the_pages_loop_structure(d, bs):
    c = small_case(seed=20 + d + bs, lens=(1, 2, 17, 40), hq=4, hkv=2, d=d, bs=bs)
    kc, vc = appended(c)
    brute = np.array(pa.decode_pseudocode_loops(wl.bits(c.q), kc, vc, c.block_tables.numpy(),
                                                c.context_lens.numpy(), c.scale))
    np.testing.assert_allclose(run_decode(c), brute, rtol=0, atol=1e-12)


def test_reductions_of_long_context_use_fp64():
    # 1% of K rows x8 stresses the softmax range; the result must still equal
    # the library routine to fp64 rounding.
    c = wl.make_case("long_small", 15, [3000, 1200], 4, 2, 64, 16, append=False,
                     k_outlier_frac=0.01)
    np.testing.assert_allclose(run_decode(c), sdpa_reference(c), rtol=0, atol=1e-11)


# ---------------------------------------------------------------------------
# 6. the append: slots, skips, bounds; ties the allocator's slot to the gather
# ---------------------------------------------------------------------------

def test_append_lands_where_the_block_table_says():
    c = small_case(seed=16, lens=(0, 1, 15, 16, 31, 32, 33))
    kc0, vc0 = wl.bits(c.k_cache), wl.bits(c.v_cache)
    kc, vc = appended(c)
    kn, vn = wl.bits(c.k_new), wl.bits(c.v_new)
    bt, cl = c.block_tables.numpy(), c.context_lens.numpy()
    touched = np.zeros(kc.shape[:2], bool)
    for b in range(c.batch):
        krows = pa.gather_sequence(kc, bt[b], int(cl[b]))
        vrows = pa.gather_sequence(vc, bt[b], int(cl[b]))
        np.testing.assert_array_equal(krows[-1], kn[b])
        np.testing.assert_array_equal(vrows[-1], vn[b])
        s = int(c.slot_mapping[b])
        touched[s // c.block_size, s % c.block_size] = True
    np.testing.assert_array_equal(kc[~touched], kc0[~touched])
    np.testing.assert_array_equal(vc[~touched], vc0[~touched])


def test_append_skips_negative_slots_and_rejects_out_of_pool():
    c = small_case(seed=17, lens=(3, 4))
    kc0, vc0 = wl.bits(c.k_cache), wl.bits(c.v_cache)
    kn, vn = wl.bits(c.k_new), wl.bits(c.v_new)
    kc, vc = pa.kv_append(kc0, vc0, kn, vn, np.array([-1, -5]))
    np.testing.assert_array_equal(kc, kc0)
    np.testing.assert_array_equal(vc, vc0)
    with pytest.raises(IndexError):
        pa.kv_append(kc0, vc0, kn, vn, np.array([0, kc0.shape[0] * kc0.shape[1]]))


# ---------------------------------------------------------------------------
# 7. the pins reject plausible mistakes (planted in copies of the oracle)
# ---------------------------------------------------------------------------

def _mutant_decode(kind):
    def fn(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None):
        hq, hkv = q.shape[1], k_cache.shape[2]
        G = hq // hkv
        bs = k_cache.shape[1]
        out = np.zeros(q.shape, np.float64)
        for b in range(q.shape[0]):
            ctx = int(context_lens[b])
            if ctx == 0:
                continue
            n = -(-ctx // bs)
            if kind == "no_mask":
                n_rows = n * bs
            else:
                n_rows = ctx
            phys = np.asarray(block_tables[b][:n], np.int64)
            K = pa.bf16_bits_to_f64(k_cache[phys].reshape(n * bs, hkv, -1)[:n_rows])
            V = pa.bf16_bits_to_f64(v_cache[phys].reshape(n * bs, hkv, -1)[:n_rows])
            if kind == "wrong_offset":
                K = pa.bf16_bits_to_f64(k_cache[phys][:, ::-1].reshape(n * bs, hkv, -1)[:ctx])
            qb = pa.bf16_bits_to_f64(q[b])
            for h in range(hq):
                kvh = (h % hkv) if kind == "strided_gqa" else h // G
                sc = 1.0 if kind == "no_scale" else scale
                s = sc * (K[:, kvh, :] @ qb[h])
                if kind == "transposed":
                    s = sc * (K[:, kvh, :].T @ K[:, kvh, :] @ qb[h])[:1].repeat(len(s))
                p = np.exp(s - np.nanmax(s))
                if kind == "no_normalise":
                    out[b, h] = p @ V[:, kvh, :]
                else:
                    out[b, h] = (p @ V[:, kvh, :]) / p.sum()
        return out
    return fn


@pytest.mark.filterwarnings("ignore:All-NaN slice")  # "no_mask" reads NaN-poisoned rows
@pytest.mark.parametrize("kind", ["strided_gqa", "no_scale", "no_mask", "wrong_offset",
                                  "transposed", "no_normalise"])
def test_pins_catch_planted_mistakes(kind):
    c = small_case(seed=30, lens=(3, 17, 40), hq=4, hkv=2, d=16, bs=8)
    ref = sdpa_reference(c)
    kc, vc = appended(c)
    bad = _mutant_decode(kind)(wl.bits(c.q), kc, vc, c.block_tables.numpy(),
                               c.context_lens.numpy(), c.scale)
    good = _mutant_decode("none")(wl.bits(c.q), kc, vc, c.block_tables.numpy(),
                                  c.context_lens.numpy(), c.scale)
    np.testing.assert_allclose(good, ref, rtol=0, atol=1e-12)     # the copy itself is right
    with np.errstate(invalid="ignore"):
        assert not np.allclose(bad, ref, rtol=0, atol=1e-6, equal_nan=False), kind
