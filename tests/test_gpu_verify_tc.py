"""GPU parity for short query chunks (speculative verification: a few query
tokens per sequence) through pa_decode_multi (bf16 pools: the persistent
tcgen05 kernel with the keys on the MMA's M side, pa_verify_tc.cu) and
pa_decode_multi_fp8 (e4m3 pools: the column-warp kernel), against the fp64
oracle's causal attention.

The tcgen05 kernel takes head_dim 128, block sizes from 8, at most 32 (token,
head) columns per KV head and splits of 128 tokens; the cases cover query groups
that fill the 32 columns and ones that leave padding columns (G = 6, ragged
token counts), block sizes 8..256 (a 128-key tile spanning 16 blocks, one
block, or part of one), splits 128..1024 with the log-sum-exp reduce, pools
whose unowned slots hold NaN (masked keys and zeroed V rows keep them out),
rows before position 0, table entries outside the pool, repeatability, a
seeded sweep of random shapes, and the speculative-verification batch of the
bench (70B heads, 4 new tokens, split 1024) with every row checked, and a
persistent launch whose blocks each walk many units (several hundred
sequences of mixed lengths and token counts); and the balanced schedule
(pa_decode_multi_balanced) on the same kernel: units cut across blocks and
merged in the kernel, sequences without query rows, rows above max_q_len.
Tolerance: the parity bar of the bf16 path (max abs <= 2e-2, per-row
relative L2 <= 5e-3).
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

POOLS = ["bf16", "e4m3"]


@pytest.fixture(autouse=True)
def _tcgen05_kernel(monkeypatch):
    monkeypatch.delenv("PA_MULTI_KERNEL", raising=False)


def run(b, case, pool, split=0, context_lens=None, block_tables=None, seed=3):
    """Append the case's new rows, run the multi-token attention; returns
    (out, the oracle's result)."""
    cl = case.context_lens if context_lens is None else context_lens
    bt = case.block_tables if block_tables is None else block_tables
    if pool == "bf16":
        k, v = case.k_cache.cuda(), case.v_cache.cuda()
        b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v)
        out = b.decode_multi(case.q.cuda(), k, v, bt.cuda(), cl.cuda(), case.q_start.cuda(),
                             case.max_q_len, case.scale, split_tokens=split)
        torch.cuda.synchronize()
        kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                              wl.bits(case.v_new), case.slot_mapping.numpy())
        return out, (kc, vc, None)
    f8 = wl.fp8_pool(case, seed)
    k, v = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    b.pa_kv_append_fp8(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v,
                       ks, vs)
    out = b.decode_multi_fp8(case.q.cuda(), k, v, ks, vs, bt.cuda(), cl.cuda(),
                             case.q_start.cuda(), case.max_q_len, case.scale,
                             split_tokens=split)
    torch.cuda.synchronize()
    kc, vc = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    pa.kv_append_fp8_inplace(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new),
                             case.slot_mapping.numpy(), f8["k_scale"].numpy(),
                             f8["v_scale"].numpy())
    assert np.array_equal(k.cpu().numpy(), kc) and np.array_equal(v.cpu().numpy(), vc)
    return out, (kc, vc, f8)


def want(case, pools, context_lens=None, block_tables=None, rows=None):
    kc, vc, f8 = pools
    cl = (case.context_lens if context_lens is None else context_lens).numpy()
    bt = (case.block_tables if block_tables is None else block_tables).numpy()
    q = wl.bits(case.q)
    if f8 is None:
        return oracle.decode_multi(q, kc, vc, bt, cl, case.q_start.numpy(), case.scale)
    return pa.decode_multi_fp8(q, kc, vc, f8["k_scale"].numpy(), f8["v_scale"].numpy(), bt, cl,
                               case.q_start.numpy(), case.scale)


SHAPES = [
    # hq, hkv, bs, ctx before, new tokens
    (64, 8, 16, [0, 100, 1000, 7, 300, 129], [4, 4, 3, 1, 2, 4]),   # G 8: 32 columns
    (32, 8, 8, [5, 0, 260, 127], [8, 3, 8, 1]),                     # G 4, block_size 8
    (8, 8, 32, [40, 0, 500], [32, 17, 9]),                          # G 1: 32 tokens
    (12, 2, 64, [50, 0, 333], [5, 2, 4]),                           # G 6: 30 columns, padding
    (16, 2, 128, [0, 200, 1111], [4, 3, 2]),                        # a block per 128-key tile
    (16, 2, 256, [100, 0, 600], [4, 1, 3]),                         # a tile inside one block
    (8, 1, 16, [10, 300, 2000], [4, 4, 4]),                         # one KV head
]


@pytest.mark.parametrize("pool", POOLS)
@pytest.mark.parametrize("hq,hkv,bs,ctx0,qlens", SHAPES)
def test_short_chunks_match_oracle(cuda_lib, pool, hq, hkv, bs, ctx0, qlens):
    case = wl.make_multi_case("vtc", 21 + hq + bs + len(ctx0), ctx0, qlens, hq, hkv, 128, bs)
    out, pools = run(cuda_lib, case, pool)
    P.assert_close(P.to_f64(out), want(case, pools), f"{pool} G={hq // hkv} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0


@pytest.mark.parametrize("pool", POOLS)
@pytest.mark.parametrize("split", [128, 256, 512, 1024])
def test_context_splits_match_oracle(cuda_lib, pool, split):
    case = wl.make_multi_case("vtcs", 40 + split, [0, 3, 127, 128, 300, 1000, 2500, 33],
                              [4, 2, 1, 4, 1, 4, 3, 4], 64, 8, 128, 16)
    out, pools = run(cuda_lib, case, pool, split=split)
    P.assert_close(P.to_f64(out), want(case, pools), f"{pool} split {split}")
    assert cuda_lib.pa_last_device_error() == 0


@pytest.mark.parametrize("pool", POOLS)
def test_rows_before_position_zero_are_zero(cuda_lib, pool):
    case = wl.make_multi_case("vtcz", 6, [0, 40], [8, 8], 16, 4, 128, 16)   # G 4: 32 columns
    short = case.context_lens.clone()
    short[0] = 5                                 # tokens 0..2 of sequence 0 sit before 0
    out, pools = run(cuda_lib, case, pool, context_lens=short)
    got = P.to_f64(out)
    assert not got[:3].any()
    P.assert_close(got, want(case, pools, context_lens=short), f"{pool} rows before position 0")


@pytest.mark.parametrize("pool", POOLS)
@pytest.mark.parametrize("split", [0, 128])
def test_block_ids_outside_the_pool_read_zeros(cuda_lib, pool, split):
    case = wl.make_multi_case("vtcoob", 17, [300, 40], [4, 4], 64, 8, 128, 16)
    nb = case.num_blocks
    bt = case.block_tables.clone()
    bt[0, 3] = nb + 7                            # keys 48..63 of sequence 0
    out, (kc, vc, f8) = run(cuda_lib, case, pool, split=split, block_tables=bt)
    assert cuda_lib.pa_last_device_error() == 0
    kz = np.concatenate([kc, np.zeros_like(kc[:1])])   # block nb: all zeros
    vz = np.concatenate([vc, np.zeros_like(vc[:1])])
    bt_ref = bt.clone()
    bt_ref[0, 3] = nb
    P.assert_close(P.to_f64(out), want(case, (kz, vz, f8), block_tables=bt_ref),
                   f"{pool} block id outside the pool")


@pytest.mark.parametrize("pool", POOLS)
def test_repeatable_bit_for_bit(cuda_lib, pool):
    case = wl.make_multi_case("vtcr", 10, [500, 20, 3000], [4, 3, 4], 64, 8, 128, 16)
    a, _ = run(cuda_lib, case, pool, split=256)
    b_, _ = run(cuda_lib, case, pool, split=256)
    assert torch.equal(a.view(torch.int16), b_.view(torch.int16))


def _random_shapes(n):
    rng = np.random.default_rng(5150)
    out = []
    for i in range(n):
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.integers(1, 9))
        bs = int(rng.choice([8, 16, 32, 64, 128, 256]))
        split = int(rng.choice([0, 128, 256, 512]))
        B = int(rng.integers(1, 7))
        ctx0 = [int(x) for x in rng.integers(0, 3000, B)]
        qlens = [int(x) for x in rng.integers(1, 32 // g + 1, B)]
        out.append((i, g * hkv, hkv, bs, split, ctx0, qlens))
    return out


@pytest.mark.parametrize("pool", POOLS)
@pytest.mark.parametrize("i,hq,hkv,bs,split,ctx0,qlens", _random_shapes(10))
def test_random_shapes_match_oracle(cuda_lib, pool, i, hq, hkv, bs, split, ctx0, qlens):
    case = wl.make_multi_case("vtcrand", 900 + i, ctx0, qlens, hq, hkv, 128, bs)
    out, pools = run(cuda_lib, case, pool, split=split, seed=11 + i)
    P.assert_close(P.to_f64(out), want(case, pools),
                   f"{pool} random shape {i}: G={hq // hkv} bs={bs} split={split}")
    assert cuda_lib.pa_last_device_error() == 0


@pytest.mark.parametrize("pool", POOLS)
def test_speculative_verify_bench_batch_every_row(cuda_lib, pool):
    # the bench's speculative-verification step (70B heads, 4 new tokens after
    # log-uniform [128, 8192] contexts, split 1024) on 64 sequences
    case = wl.spec_verify_case(seed=2, batch=64, q_len=4)
    out, pools = run(cuda_lib, case, pool, split=1024)
    P.assert_close(P.to_f64(out), want(case, pools), f"{pool} spec verify, split 1024")
    assert cuda_lib.pa_last_device_error() == 0


@pytest.mark.parametrize("pool", POOLS)
def test_persistent_blocks_walk_many_units(cuda_lib, pool):
    # 300 sequences x 8 KV heads x up to 6 splits: every block of the
    # persistent launch takes many units, short and long, with and without a
    # key in its split, some with nothing to attend (rows before position 0)
    rng = np.random.default_rng(77)
    ctx0 = [int(x) for x in rng.integers(0, 1500, 300)]
    qlens = [int(x) for x in rng.integers(1, 5, 300)]
    case = wl.make_multi_case("vtcmany", 55, ctx0, qlens, 64, 8, 128, 16)
    short = case.context_lens.clone()
    short[::37] = 2                              # rows before position 0 in some sequences
    short = torch.maximum(short, torch.ones_like(short))
    out, pools = run(cuda_lib, case, pool, split=256, context_lens=short)
    P.assert_close(P.to_f64(out), want(case, pools, context_lens=short), f"{pool} many units")
    assert cuda_lib.pa_last_device_error() == 0


def _balanced(b, case, context_lens=None, max_q_len=None, reps=2):
    cl = case.context_lens if context_lens is None else context_lens
    ws = torch.zeros(b.pa_decode_multi_balanced_workspace_bytes(case.batch, case.num_kv_heads, 128),
                     dtype=torch.uint8, device="cuda")
    k, v = case.k_cache.cuda(), case.v_cache.cuda()
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v)
    outs = []
    for _ in range(reps):                           # the workspace is reusable
        out = torch.zeros_like(case.q).cuda()
        b.pa_decode_multi_balanced(case.q.cuda(), k, v, case.block_tables.cuda(), cl.cuda(),
                                   case.q_start.cuda(), max_q_len or case.max_q_len, case.scale,
                                   ws, out)
        outs.append(out)
    torch.cuda.synchronize()
    counters = ws[: case.batch * case.num_kv_heads * 8 * 4].view(torch.int32)
    assert torch.all(counters == 0)                 # the tickets are left zero
    return outs


@pytest.mark.parametrize("split_heads", [(64, 8), (16, 2), (8, 1)])
def test_balanced_schedule_many_units(cuda_lib, split_heads):
    # the balanced schedule on the tcgen05 kernel: every block an equal range
    # of 128-key tiles, units cut across blocks merged in the kernel, long
    # and short contexts, sequences without query rows, rows before position 0
    hq, hkv = split_heads
    g = hq // hkv
    rng = np.random.default_rng(91 + hq)
    B = 260
    ctx0 = [int(x) for x in np.exp(rng.uniform(np.log(1), np.log(20000), B))]
    qlens = [int(x) for x in rng.integers(0, min(4, 32 // g) + 1, B)]
    qlens[0] = min(4, 32 // g)
    case = wl.make_multi_case("vtcbal", 31 + hq, ctx0, qlens, hq, hkv, 128, 16)
    short = case.context_lens.clone()
    short[5::41] = 1                                # rows before position 0
    short = torch.maximum(short, torch.ones_like(short))
    a, b_ = _balanced(cuda_lib, case, context_lens=short)
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), case.slot_mapping.numpy())
    want_ = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                                short.numpy(), case.q_start.numpy(), case.scale)
    P.assert_close(P.to_f64(a), want_, f"balanced tcgen05 G={g}")
    assert torch.equal(a.view(torch.int16), b_.view(torch.int16))
    assert cuda_lib.pa_last_device_error() == 0


def test_balanced_schedule_rows_above_max_q_len(cuda_lib):
    # a sequence with more rows than max_q_len holds no tiles, is left as it
    # is and sets bit 16; the others are attended as usual
    case = wl.make_multi_case("vtcbalbad", 13, [3000, 100, 50], [6, 3, 4], 64, 8, 128, 16)
    out, = _balanced(cuda_lib, case, max_q_len=4, reps=1)
    assert cuda_lib.pa_last_device_error() & 16
    got = P.to_f64(out)
    assert not got[:6].any()
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), case.slot_mapping.numpy())
    want_ = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                                case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    P.assert_close(got[6:], want_[6:], "balanced tcgen05, the other sequences")
