"""GPU parity for long query chunks over an e4m3 pool: the tcgen05 prefill
kernel with the e4m3 rows widened to f16 in shared memory, through
pa_decode_multi_fp8, against the oracle's causal attention over the
read-back pool (value(code) * scale of the head).

Covers query groups that divide the 256-row block and one that leaves
padding rows (G = 6), block sizes 1..256 (rows gathered by cp.async below
8, TMA boxes from 8), chunks spanning many 128-key tiles
with ragged tails, pools whose unowned slots hold NaN codes (masked keys and
zeroed V rows must keep them out), rows before position 0, a seeded sweep of
random shapes, and the chunked-prefill bench step (8 x 2048 new tokens after
6144 cached, 64/8 heads) on sampled rows. Tolerance: the parity bar of the
bf16 path (max abs <= 2e-2, per-row relative L2 <= 5e-3).
"""

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


def pools(case, seed):
    f8 = wl.fp8_pool(case, seed)
    kc, vc = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    pa.kv_append_fp8_inplace(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new),
                             case.slot_mapping.numpy(), f8["k_scale"].numpy(),
                             f8["v_scale"].numpy())
    return f8, kc, vc


def run(b, case, f8, context_lens=None):
    k, v = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    b.pa_kv_append_fp8(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v,
                       ks, vs)
    cl = case.context_lens if context_lens is None else context_lens
    out = b.decode_multi_fp8(case.q.cuda(), k, v, ks, vs, case.block_tables.cuda(), cl.cuda(),
                             case.q_start.cuda(), case.max_q_len, case.scale)
    torch.cuda.synchronize()
    return out, k, v


def want(case, f8, kc, vc, context_lens=None):
    cl = case.context_lens if context_lens is None else context_lens
    return pa.decode_multi_fp8(wl.bits(case.q), kc, vc, f8["k_scale"].numpy(),
                               f8["v_scale"].numpy(), case.block_tables.numpy(), cl.numpy(),
                               case.q_start.numpy(), case.scale)


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
def test_e4m3_long_chunks_match_oracle(cuda_lib, hq, hkv, bs, ctx0, qlens):
    case = wl.make_multi_case("tc8", 31 + hq + bs + len(ctx0), ctx0, qlens, hq, hkv, 128, bs)
    f8, kc, vc = pools(case, 3)
    out, k, v = run(cuda_lib, case, f8)
    assert np.array_equal(k.cpu().numpy(), kc) and np.array_equal(v.cpu().numpy(), vc)
    P.assert_close(P.to_f64(out), want(case, f8, kc, vc), f"e4m3 G={hq // hkv} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0


def test_e4m3_rows_before_position_zero_are_zero(cuda_lib):
    case = wl.make_multi_case("tc8z", 6, [0, 40], [200, 150], 16, 2, 128, 16)
    f8, kc, vc = pools(case, 4)
    short = case.context_lens.clone()
    short[0] = 130                               # tokens 0..69 of sequence 0 sit before 0
    out, _, _ = run(cuda_lib, case, f8, context_lens=short)
    got = P.to_f64(out)
    assert not got[:70].any()
    P.assert_close(got, want(case, f8, kc, vc, short), "e4m3 rows before position 0")


def test_e4m3_repeatable_bit_for_bit(cuda_lib):
    case = wl.make_multi_case("tc8r", 10, [500, 20], [400, 333], 64, 8, 128, 16)
    f8, _, _ = pools(case, 5)
    a, _, _ = run(cuda_lib, case, f8)
    b_, _, _ = run(cuda_lib, case, f8)
    assert torch.equal(a.view(torch.int16), b_.view(torch.int16))


def test_e4m3_long_chunks_with_splits_are_refused(cuda_lib):
    b = cuda_lib
    case = wl.make_multi_case("tc8u", 12, [10, 40], [100, 90], 16, 2, 128, 16)
    f8, _, _ = pools(case, 6)
    k, v = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    R = int(case.q.shape[0])
    out = torch.zeros_like(case.q).cuda()
    S = 8
    po = torch.empty((R, 16, S, 128), dtype=torch.float32, device="cuda")
    pl = torch.empty((R, 16, S), dtype=torch.float32, device="cuda")
    rl = torch.empty(R, dtype=torch.int32, device="cuda")
    with pytest.raises(b.PagedKVError) as e:      # long chunks run unsplit only
        b.pa_decode_multi_fp8(case.q.cuda(), k, v, ks, vs, case.block_tables.cuda(),
                              case.context_lens.cuda(), case.q_start.cuda(), case.max_q_len,
                              case.scale, out, 32, S, po, pl, rl)
    assert e.value.status == -2


def _random_shapes(n):
    rng = np.random.default_rng(4048)
    out = []
    for i in range(n):
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.integers(1, 9))
        bs = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 256]))
        B = int(rng.integers(1, 5))
        ctx0 = [int(x) for x in rng.integers(0, 900, B)]
        qlens = [int(x) for x in rng.integers(1, 400, B)]
        qlens[0] = max(qlens[0], 80 // g + 1)      # at least one long chunk: > 64 rows
        out.append((i, g * hkv, hkv, bs, ctx0, qlens))
    return out


@pytest.mark.parametrize("i,hq,hkv,bs,ctx0,qlens", _random_shapes(10))
def test_e4m3_random_shapes_match_oracle(cuda_lib, i, hq, hkv, bs, ctx0, qlens):
    case = wl.make_multi_case("tc8rand", 700 + i, ctx0, qlens, hq, hkv, 128, bs)
    f8, kc, vc = pools(case, 7 + i)
    out, _, _ = run(cuda_lib, case, f8)
    P.assert_close(P.to_f64(out), want(case, f8, kc, vc),
                   f"e4m3 random shape {i}: G={hq // hkv} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0


def test_e4m3_prefill_bench_step_on_sampled_rows(cuda_lib):
    # the bench's chunked-prefill step over an e4m3 pool: 8 sequences, 2048
    # new tokens after 6144 cached, 64 q heads / 8 KV heads; rows sampled
    # across every sequence, each checked alone
    case = wl.make_multi_case("prefill", 0, [6144] * 8, [2048] * 8, 64, 8, 128, 16)
    f8, kc, vc = pools(case, 0)
    out, _, _ = run(cuda_lib, case, f8)
    out = P.to_f64(out)
    q = wl.bits(case.q)
    bt = case.block_tables.numpy()
    ks, vs = f8["k_scale"].numpy(), f8["v_scale"].numpy()
    rng = np.random.default_rng(6)
    for s in range(8):
        picks = sorted({0, 1, 31, 32, 127, 128, 2047} | set(rng.integers(0, 2048, 3).tolist()))
        for i in picks:
            row = s * 2048 + i
            w = pa.decode_multi_fp8(q[row:row + 1], kc, vc, ks, vs, bt[s:s + 1],
                                    np.array([6144 + i + 1]), np.array([0, 1]), case.scale)
            P.assert_close(out[row:row + 1], w, f"e4m3 sequence {s} token {i}")
    assert cuda_lib.pa_last_device_error() == 0
