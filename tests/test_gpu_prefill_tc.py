"""GPU parity for long query chunks (chunked prefill) on the tcgen05 kernel of
pa_decode_multi, and on the mma.sync row-block kernel it replaces
(PA_PREFILL_KERNEL=rowblock), against the fp64 oracle's causal attention.

Covers head_dim 128 and 64, query groups that divide the 256-row block and
ones that leave padding rows (G = 6), block sizes 1..256 (rows gathered by
cp.async below 8, one TMA box per block from 8, a 128-key tile inside one
block from 128), chunks spanning many 128-key
tiles with ragged tails, cached prefixes that are not tile multiples, pools
whose unowned slots are NaN (masked keys and zeroed V rows must keep them
out), rows before position 0, repeatability, and the chunked-prefill bench
step (8 x 2048 new tokens after 6144 cached, 64/8 heads) on sampled rows.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

KERNELS = ["tcgen05", "rowblock"]


@pytest.fixture(params=KERNELS)
def kernel(request, monkeypatch):
    if request.param == "rowblock":
        monkeypatch.setenv("PA_PREFILL_KERNEL", "rowblock")
    else:
        monkeypatch.delenv("PA_PREFILL_KERNEL", raising=False)
    return request.param


def appended(case):
    return pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                        wl.bits(case.v_new), case.slot_mapping.numpy())


def run(b, case, context_lens=None):
    k, v = case.k_cache.cuda(), case.v_cache.cuda()
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v)
    cl = case.context_lens if context_lens is None else context_lens
    out = b.decode_multi(case.q.cuda(), k, v, case.block_tables.cuda(), cl.cuda(),
                         case.q_start.cuda(), case.max_q_len, case.scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("hq,hkv,bs,ctx0,qlens", [
    (64, 8, 16, [0, 100, 1000, 7], [300, 129, 40, 257]),      # G 8: 32 tokens a block
    (8, 8, 16, [0, 250], [600, 513]),                          # G 1: 256 tokens a block
    (32, 8, 32, [3, 0, 129], [130, 77, 200]),                  # G 4
    (12, 2, 16, [50, 0], [90, 43]),                            # G 6: 42 tokens, 4 padding rows
    (8, 1, 64, [10, 300], [5, 30]),                            # one KV head, block_size 64
    (16, 2, 8, [0, 31], [100, 70]),                            # block_size 8
    (16, 2, 128, [0, 200], [160, 300]),                        # one block per 128-key tile
    (16, 2, 256, [100, 0, 600], [200, 90, 40]),                # a tile inside one block
    (16, 2, 4, [0, 37], [130, 90]),                            # block_size 4 (cp.async rows)
    (64, 8, 2, [5, 0], [70, 33]),                              # block_size 2
    (12, 2, 1, [50, 0], [90, 43]),                             # block_size 1, G 6
])
def test_long_chunks_match_oracle(cuda_lib, kernel, hq, hkv, bs, ctx0, qlens):
    case = wl.make_multi_case("tc", 7 + hq + bs + len(ctx0), ctx0, qlens, hq, hkv, 128, bs)
    out = run(cuda_lib, case)
    kc, vc = appended(case)
    want = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    P.assert_close(P.to_f64(out), want, f"{kernel} G={hq // hkv} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0


@pytest.mark.parametrize("hq,hkv,bs,ctx0,qlens", [
    (32, 4, 16, [0, 100, 1000, 7], [300, 129, 40, 257]),      # G 8
    (8, 8, 8, [0, 250], [600, 513]),                           # G 1, block_size 8
    (12, 2, 64, [50, 0], [90, 43]),                            # G 6, padding rows
    (16, 2, 256, [100, 0, 600], [200, 90, 40]),                # a tile inside one block
    (16, 2, 2, [0, 31], [150, 70]),                            # block_size 2 (cp.async rows)
])
def test_head_dim_64_long_chunks_match_oracle(cuda_lib, kernel, hq, hkv, bs, ctx0, qlens):
    case = wl.make_multi_case("tc64", 11 + hq + bs, ctx0, qlens, hq, hkv, 64, bs)
    out = run(cuda_lib, case)
    kc, vc = appended(case)
    want = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    P.assert_close(P.to_f64(out), want, f"{kernel} D=64 G={hq // hkv} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0


def test_rows_before_position_zero_are_zero(cuda_lib, kernel):
    # a context shorter than the chunk: the first rows have no position
    case = wl.make_multi_case("tcz", 5, [0, 40], [200, 150], 16, 2, 128, 16)
    short = case.context_lens.clone()
    short[0] = 130                               # tokens 0..69 of sequence 0 sit before 0
    out = run(cuda_lib, case, context_lens=short)
    kc, vc = appended(case)
    want = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               short.numpy(), case.q_start.numpy(), case.scale)
    got = P.to_f64(out)
    assert not got[:70].any()
    P.assert_close(got, want, f"{kernel} rows before position 0")


def test_repeatable_bit_for_bit(cuda_lib):
    case = wl.make_multi_case("tcr", 9, [500, 20], [400, 333], 64, 8, 128, 16)
    a = run(cuda_lib, case)
    b_ = run(cuda_lib, case)
    assert torch.equal(a.view(torch.int16), b_.view(torch.int16))


def test_prefill_bench_step_on_sampled_rows(cuda_lib):
    # the bench's chunked-prefill step: 8 sequences, 2048 new tokens after
    # 6144 cached, 64 q heads / 8 KV heads; rows sampled across every
    # sequence (first, diagonal-tile and last tokens), each checked alone
    case = wl.make_multi_case("prefill", 0, [6144] * 8, [2048] * 8, 64, 8, 128, 16)
    out = P.to_f64(run(cuda_lib, case))
    kc, vc = appended(case)
    q = wl.bits(case.q)
    bt = case.block_tables.numpy()
    rng = np.random.default_rng(5)
    for s in range(8):
        picks = sorted({0, 1, 31, 32, 127, 128, 2047} | set(rng.integers(0, 2048, 3).tolist()))
        for i in picks:
            row = s * 2048 + i
            want = oracle.decode_multi(q[row:row + 1], kc, vc, bt[s:s + 1],
                                       np.array([6144 + i + 1]), np.array([0, 1]), case.scale)
            P.assert_close(out[row:row + 1], want, f"sequence {s} token {i}")
    assert cuda_lib.pa_last_device_error() == 0


def test_rows_above_max_q_len_set_the_shape_bit(cuda_lib, kernel):
    # long-chunk launch (max_q_len 20 x G 8 > 64 rows) with a sequence of 40
    # tokens: that sequence is skipped, the device error word gets bit 16
    b = cuda_lib
    case = wl.make_multi_case("tcshape", 13, [10, 100], [40, 12], 16, 2, 128, 16)
    k, v = case.k_cache.cuda(), case.v_cache.cuda()
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v)
    out = torch.zeros_like(case.q).cuda()
    b.pa_decode_multi(case.q.cuda(), k, v, case.block_tables.cuda(), case.context_lens.cuda(),
                      case.q_start.cuda(), 20, case.scale, out)
    torch.cuda.synchronize()
    assert b.pa_last_device_error() & 16
    got = P.to_f64(out)
    assert not got[:40].any()                    # the skipped sequence: untouched
    kc, vc = appended(case)
    want = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    P.assert_close(got[40:], want[40:], f"{kernel} the other sequence")


@pytest.mark.parametrize("bs", [16, 2])
def test_block_ids_outside_the_pool_read_zeros(cuda_lib, bs):
    # a table entry inside the context that points past the pool: the kernel
    # reads zero K/V rows there (a TMA box wholly out of range, or zero-filled
    # cp.async copies at block size 2) and faults nothing; the oracle sees the
    # same once that entry names a zero block
    b = cuda_lib
    case = wl.make_multi_case("tcoob", 17, [100, 40], [300, 90], 16, 2, 128, bs)
    nb = case.k_cache.shape[0]
    k, v = case.k_cache.cuda(), case.v_cache.cuda()
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v)
    kc, vc = appended(case)
    bt = case.block_tables.clone()
    bt[0, 3] = nb + 7                            # keys 3 bs .. 4 bs - 1 of sequence 0
    out = b.decode_multi(case.q.cuda(), k, v, bt.cuda(), case.context_lens.cuda(),
                         case.q_start.cuda(), case.max_q_len, case.scale)
    torch.cuda.synchronize()
    assert b.pa_last_device_error() == 0
    kz = np.concatenate([kc, np.zeros_like(kc[:1])])   # block nb: all zeros
    vz = np.concatenate([vc, np.zeros_like(vc[:1])])
    bt_ref = bt.numpy().copy()
    bt_ref[0, 3] = nb
    want = oracle.decode_multi(wl.bits(case.q), kz, vz, bt_ref, case.context_lens.numpy(),
                               case.q_start.numpy(), case.scale)
    P.assert_close(P.to_f64(out), want, "block id outside the pool")


def _random_shapes(n):
    rng = np.random.default_rng(2024)
    out = []
    for i in range(n):
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.integers(1, 9))
        d = int(rng.choice([64, 128]))
        bs = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256]))
        B = int(rng.integers(1, 5))
        ctx0 = [int(x) for x in rng.integers(0, 900, B)]
        qlens = [int(x) for x in rng.integers(1, 400, B)]
        qlens[0] = max(qlens[0], 80 // g + 1)      # at least one long chunk: > 64 rows
        out.append((i, g * hkv, hkv, d, bs, ctx0, qlens))
    return out


@pytest.mark.parametrize("i,hq,hkv,d,bs,ctx0,qlens", _random_shapes(12))
def test_random_shapes_match_oracle(cuda_lib, i, hq, hkv, d, bs, ctx0, qlens):
    case = wl.make_multi_case("tcrand", 500 + i, ctx0, qlens, hq, hkv, d, bs)
    out = run(cuda_lib, case)
    kc, vc = appended(case)
    want = oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    P.assert_close(P.to_f64(out), want, f"random shape {i}: G={hq // hkv} D={d} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0
