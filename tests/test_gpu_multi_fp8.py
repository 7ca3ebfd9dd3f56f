"""GPU parity for several query tokens per sequence over an FP8 (e4m3) pool
(pa_decode_multi_fp8) against the fp64 oracle's causal attention on the
dequantized pool (oracle.decode_multi_fp8): the appended codes bit for bit,
then ragged token counts, GQA groups up to the 64-column limit, block sizes
1..32 (cp.async and TMA loads), context splits with the reduce, the 70B-shape
speculative-verification batch, and the argument checks."""

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

CTX = [0, 1, 15, 16, 17, 31, 33, 64, 100, 257, 700]


def run_fp8(b, case, seed, split=0):
    """Append the case's new rows into an e4m3 pool on the device and run the
    multi-token attention; returns (out, oracle codes after the append, f8)."""
    f8 = wl.fp8_pool(case, seed)
    kd, vd = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    b.pa_kv_append_fp8(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), kd, vd,
                       ks, vs)
    out = b.decode_multi_fp8(case.q.cuda(), kd, vd, ks, vs, case.block_tables.cuda(),
                             case.context_lens.cuda(), case.q_start.cuda(), case.max_q_len,
                             case.scale, split_tokens=split)
    torch.cuda.synchronize()
    kc, vc = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    pa.kv_append_fp8_inplace(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new),
                             case.slot_mapping.numpy(), f8["k_scale"].numpy(),
                             f8["v_scale"].numpy())
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    return out, kc, vc, f8


def oracle_fp8(case, kc, vc, f8):
    return oracle.decode_multi_fp8(wl.bits(case.q), kc, vc, f8["k_scale"].numpy(),
                                   f8["v_scale"].numpy(), case.block_tables.numpy(),
                                   case.context_lens.numpy(), case.q_start.numpy(), case.scale)


@pytest.mark.parametrize("qlen,hq,hkv,bs", [
    (1, 8, 1, 16), (4, 64, 8, 16), (8, 64, 8, 16), (3, 8, 2, 16), (5, 16, 2, 8),
    (7, 8, 2, 1), (2, 8, 8, 32), (6, 32, 8, 16)])
def test_multi_fp8_matches_oracle(cuda_lib, qlen, hq, hkv, bs):
    rng = np.random.default_rng(qlen * 31 + hq + bs)
    qlens = [int(x) for x in rng.integers(1, qlen + 1, len(CTX))]
    qlens[0] = qlen
    case = wl.make_multi_case("mqf8", 300 + qlen + bs, CTX, qlens, hq, hkv, 128, bs)
    out, kc, vc, f8 = run_fp8(cuda_lib, case, 300 + qlen)
    P.assert_close(P.to_f64(out), oracle_fp8(case, kc, vc, f8),
                   f"e4m3 q_len<={qlen} G={hq // hkv} bs={bs}")
    assert cuda_lib.pa_last_device_error() == 0


@pytest.mark.parametrize("split", [32, 128, 256, 1024])
def test_multi_fp8_with_context_splits(cuda_lib, split):
    case = wl.make_multi_case("mqf8s", 330 + split, [0, 3, 60, 300, 1000, 33],
                              [4, 2, 8, 1, 8, 5], 64, 8, 128, 16)
    out, kc, vc, f8 = run_fp8(cuda_lib, case, 330, split=split)
    P.assert_close(P.to_f64(out), oracle_fp8(case, kc, vc, f8), f"e4m3 split {split}")


def test_multi_fp8_speculative_verify_batch(cuda_lib):
    # the spec-verify shape (70B heads, 4 new tokens, log-uniform contexts) on
    # 64 sequences, every row checked, split 1024 as the bench runs it
    case = wl.spec_verify_case(7, batch=64, q_len=4)
    out, kc, vc, f8 = run_fp8(cuda_lib, case, 7, split=1024)
    P.assert_close(P.to_f64(out), oracle_fp8(case, kc, vc, f8), "e4m3 spec verify")


def test_multi_fp8_argument_checks(cuda_lib):
    b = cuda_lib
    case = wl.make_multi_case("mqf8a", 340, [10, 20], [3, 2], 16, 2, 64, 16)
    f8 = wl.fp8_pool(case, 340)
    q = case.q.cuda()
    kd, vd = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    bt, cl, qs = case.block_tables.cuda(), case.context_lens.cuda(), case.q_start.cuda()
    out = torch.empty_like(q)
    with pytest.raises(b.PagedKVError) as e:        # head_dim 64: one e4m3 row is 128 bytes
        b.pa_decode_multi_fp8(q, kd, vd, ks, vs, bt, cl, qs, 3, case.scale, out)
    assert e.value.status == -2
    case = wl.make_multi_case("mqf8b", 341, [10, 20], [9, 2], 16, 2, 128, 16)
    f8 = wl.fp8_pool(case, 341)
    q = case.q.cuda()
    kd, vd = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    bt, cl, qs = case.block_tables.cuda(), case.context_lens.cuda(), case.q_start.cuda()
    out = torch.empty_like(q)
    S = 4
    po = torch.empty((q.shape[0], 16, S, 128), dtype=torch.float32, device="cuda")
    pl = torch.empty((q.shape[0], 16, S), dtype=torch.float32, device="cuda")
    rl = torch.empty(q.shape[0], dtype=torch.int32, device="cuda")
    # 9 tokens x 8 heads > 64 columns: a long chunk, which runs unsplit only
    with pytest.raises(b.PagedKVError) as e:
        b.pa_decode_multi_fp8(q, kd, vd, ks, vs, bt, cl, qs, 9, case.scale, out, 32, S, po,
                              pl, rl)
    assert e.value.status == -2
    with pytest.raises(b.PagedKVError) as e:        # split not a multiple of the 32-token tile
        b.pa_decode_multi_fp8(q, kd, vd, ks, vs, bt, cl, qs, 8, case.scale, out, 16, S, po,
                              pl, rl)
    assert e.value.status == -1
