"""GPU parity for several query tokens per sequence (pa_decode_multi) against
the fp64 oracle's causal attention: ragged token counts, GQA groups up to the
64-column limit, head_dim 64/128, block sizes 1..32, with and without context
splits (+ pa_decode_splitk_reduce), a prompt fed chunk by chunk, the 70B-shape
speculative-verification batch, and the argument and shape checks."""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


def run_multi(b, case, split=0):
    d = dict(q=case.q.cuda(), k=case.k_cache.cuda(), v=case.v_cache.cuda(),
             bt=case.block_tables.cuda(), cl=case.context_lens.cuda(), qs=case.q_start.cuda())
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), d["k"], d["v"])
    out = b.decode_multi(d["q"], d["k"], d["v"], d["bt"], d["cl"], d["qs"], case.max_q_len,
                         case.scale, split_tokens=split)
    torch.cuda.synchronize()
    return out


def oracle_multi(case, rows=None):
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), case.slot_mapping.numpy())
    return oracle.decode_multi(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)


CTX = [0, 1, 15, 16, 17, 40, 100, 257, 700]


@pytest.mark.parametrize("qlen,hq,hkv,d,bs", [
    (1, 8, 1, 128, 16), (4, 8, 1, 128, 16), (8, 64, 8, 128, 16), (3, 8, 2, 128, 16),
    (16, 8, 2, 64, 16), (64, 4, 4, 128, 16), (5, 16, 2, 64, 8), (7, 8, 2, 128, 1),
    (2, 8, 8, 128, 32), (6, 32, 8, 128, 16)])
def test_multi_matches_oracle(cuda_lib, multi_kernel, qlen, hq, hkv, d, bs):
    rng = np.random.default_rng(qlen * 100 + hq + bs)
    qlens = [int(x) for x in rng.integers(1, qlen + 1, len(CTX))]
    qlens[0] = qlen
    case = wl.make_multi_case("mq", 40 + qlen + bs, CTX, qlens, hq, hkv, d, bs)
    out = run_multi(cuda_lib, case)
    P.assert_close(P.to_f64(out), oracle_multi(case),
                   f"{multi_kernel} q_len<={qlen} G={hq // hkv} bs={bs}")


@pytest.mark.parametrize("qlen,hq,hkv,d,bs", [
    (1, 8, 1, 128, 16), (4, 8, 1, 128, 16), (8, 64, 8, 128, 16), (3, 8, 2, 128, 16),
    (16, 8, 2, 64, 16), (64, 4, 4, 128, 16), (5, 16, 2, 64, 8), (7, 8, 2, 128, 1),
    (2, 8, 8, 128, 32), (6, 32, 8, 128, 16)])
def test_balanced_multi_matches_oracle(cuda_lib, multi_kernel, qlen, hq, hkv, d, bs):
    rng = np.random.default_rng(qlen * 100 + hq + bs)
    qlens = [int(x) for x in rng.integers(1, qlen + 1, len(CTX))]
    qlens[0] = qlen
    case = wl.make_multi_case("mqb", 40 + qlen + bs, CTX, qlens, hq, hkv, d, bs)
    out = run_multi(cuda_lib, case, split=cuda_lib.BALANCED_MULTI)
    P.assert_close(P.to_f64(out), oracle_multi(case),
                   f"{multi_kernel} balanced q_len<={qlen} G={hq // hkv}")


@pytest.mark.parametrize("lens", [[5000, 3, 0, 700, 1], [1] * 40, [9000] * 3 + [17] * 50],
                         ids=["mixed", "tiny_units", "long_and_short"])
def test_balanced_multi_cut_units_and_sequences_without_rows(cuda_lib, multi_kernel, lens):
    # long contexts are cut across many blocks (per-column records merged in
    # the kernel); a sequence with no query rows holds no tiles
    qlens = [(i % 4) for i in range(len(lens))]
    qlens[0] = 4
    ctx0 = [max(c, 4) for c in lens]
    case = wl.make_multi_case("mqbc", 77 + len(lens), ctx0, qlens, 64, 8, 128, 16)
    b = cuda_lib
    ws = torch.zeros(b.pa_decode_multi_balanced_workspace_bytes(case.batch, 8, 128),
                     dtype=torch.uint8, device="cuda")
    d = dict(q=case.q.cuda(), k=case.k_cache.cuda(), v=case.v_cache.cuda())
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), d["k"], d["v"])
    outs = []
    for _ in range(2):                              # the workspace is reusable
        out = torch.full_like(d["q"], float("nan"))
        b.pa_decode_multi_balanced(d["q"], d["k"], d["v"], case.block_tables.cuda(),
                                   case.context_lens.cuda(), case.q_start.cuda(),
                                   case.max_q_len, case.scale, ws, out)
        outs.append(out)
    torch.cuda.synchronize()
    P.assert_close(P.to_f64(outs[0]), oracle_multi(case), f"{multi_kernel} balanced cut units")
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    counters = ws[: case.batch * 8 * 8 * 4].view(torch.int32)
    assert torch.all(counters == 0)
    assert b.pa_last_device_error() == 0


@pytest.mark.parametrize("qmax,hq,hkv,d,bs", [
    (9, 8, 1, 128, 16), (40, 64, 8, 128, 16), (300, 8, 1, 128, 16), (100, 16, 4, 64, 16),
    (70, 8, 2, 128, 8), (33, 8, 2, 128, 1), (65, 2, 2, 128, 32)])
def test_long_chunks_match_oracle(cuda_lib, qmax, hq, hkv, d, bs):
    # more (token, head) rows than 64: the row-block kernel, every sequence of
    # the batch (short ones too) on it
    rng = np.random.default_rng(qmax + hq + bs)
    ctx0 = [0, 5, 17, 200, 1000, 3]
    qlens = [int(x) for x in rng.integers(1, qmax + 1, len(ctx0))]
    qlens[0] = qmax
    case = wl.make_multi_case("long", 90 + qmax, ctx0, qlens, hq, hkv, d, bs)
    out = run_multi(cuda_lib, case)
    P.assert_close(P.to_f64(out), oracle_multi(case), f"chunk <= {qmax}, G={hq // hkv}")


def test_long_prompt_in_large_chunks_equals_full_causal_attention(cuda_lib):
    b = cuda_lib
    n, hq, hkv, d, bs = 700, 64, 8, 128, 16
    full = wl.make_multi_case("bigchunks", 62, [0], [n], hq, hkv, d, bs)
    k, v = full.k_cache.cuda(), full.v_cache.cuda()
    bt = full.block_tables.cuda()
    kc, vc = pa.kv_append(wl.bits(full.k_cache), wl.bits(full.v_cache), wl.bits(full.k_new),
                          wl.bits(full.v_new), full.slot_mapping.numpy())
    sub = list(range(0, n, 7)) + [n - 1]
    want = oracle.decode_multi(wl.bits(full.q), kc, vc, full.block_tables.numpy(),
                               np.array([n]), np.array([0, n]), full.scale)
    got = np.zeros_like(want)
    a = 0
    for c in [256, 5, 256, 183]:
        sl = slice(a, a + c)
        b.pa_kv_append(full.k_new[sl].cuda(), full.v_new[sl].cuda(),
                       full.slot_mapping[sl].cuda(), k, v)
        out = b.decode_multi(full.q[sl].cuda(), k, v, bt,
                             torch.tensor([a + c], dtype=torch.int32, device="cuda"),
                             torch.tensor([0, c], dtype=torch.int32, device="cuda"), c,
                             full.scale)
        torch.cuda.synchronize()
        got[sl] = P.to_f64(out)
        a += c
    P.assert_close(got[sub], want[sub], "4 chunks of a 700-token prompt")


def test_long_chunks_refuse_context_splits(cuda_lib):
    b = cuda_lib
    case = wl.make_multi_case("ls", 63, [10], [20], 64, 8, 128, 16)
    with pytest.raises(b.PagedKVError) as e:
        run_multi(b, case, split=64)
    assert e.value.status == -2


@pytest.mark.parametrize("split", [16, 64, 128, 256, 1024])
def test_multi_with_context_splits(cuda_lib, multi_kernel, split):
    case = wl.make_multi_case("mqs", 50 + split, [0, 3, 60, 300, 1000, 33], [4, 2, 8, 1, 8, 5],
                              64, 8, 128, 16)
    out = run_multi(cuda_lib, case, split=split)
    P.assert_close(P.to_f64(out), oracle_multi(case), f"{multi_kernel} split {split}")


def test_prompt_fed_chunk_by_chunk_equals_full_causal_attention(cuda_lib, multi_kernel):
    b = cuda_lib
    n, hq, hkv, d, bs = 96, 16, 2, 128, 16
    full = wl.make_multi_case("chunks", 61, [0], [n], hq, hkv, d, bs)
    k, v = full.k_cache.cuda(), full.v_cache.cuda()
    bt = full.block_tables.cuda()
    kc, vc = pa.kv_append(wl.bits(full.k_cache), wl.bits(full.v_cache), wl.bits(full.k_new),
                          wl.bits(full.v_new), full.slot_mapping.numpy())
    want = oracle.decode_multi(wl.bits(full.q), kc, vc, full.block_tables.numpy(),
                               np.array([n]), np.array([0, n]), full.scale)
    a = 0
    for c in [8, 1, 7, 8, 8, 8, 8, 4, 4, 8, 8, 8, 8, 8]:   # at most 64 // G tokens a call
        sl = slice(a, a + c)
        b.pa_kv_append(full.k_new[sl].cuda(), full.v_new[sl].cuda(),
                       full.slot_mapping[sl].cuda(), k, v)
        out = b.decode_multi(full.q[sl].cuda(), k, v, bt,
                             torch.tensor([a + c], dtype=torch.int32, device="cuda"),
                             torch.tensor([0, c], dtype=torch.int32, device="cuda"), c,
                             full.scale)
        torch.cuda.synchronize()
        P.assert_close(P.to_f64(out), want[sl], f"chunk at {a}")
        a += c
    assert a == n


@pytest.mark.parametrize("schedule", ["unsplit", "split1024", "balanced"])
def test_speculative_verify_70b_shape_sampled(cuda_lib, multi_kernel, schedule):
    case = wl.spec_verify_case(seed=0, batch=256, q_len=4)
    split = {"unsplit": 0, "split1024": 1024, "balanced": cuda_lib.BALANCED_MULTI}[schedule]
    out = P.to_f64(run_multi(cuda_lib, case, split=split))
    sub = [0, 17, 101, 199, 255]
    qs = case.q_start.numpy()
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), case.slot_mapping.numpy())
    q_rows = np.concatenate([wl.bits(case.q)[qs[s]:qs[s + 1]] for s in sub])
    starts = np.concatenate([[0], np.cumsum([qs[s + 1] - qs[s] for s in sub])])
    want = oracle.decode_multi(q_rows, kc, vc, case.block_tables.numpy()[sub],
                               case.context_lens.numpy()[sub], starts, case.scale)
    got = np.concatenate([out[qs[s]:qs[s + 1]] for s in sub])
    P.assert_close(got, want, f"70B spec verify, {multi_kernel}, {schedule}")
    assert np.isfinite(out).all()


def test_multi_argument_checks(cuda_lib):
    b = cuda_lib
    case = wl.make_multi_case("chk", 70, [5, 9], [2, 3], 16, 2, 128, 16)
    q, k, v = case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda()
    bt, cl, qs = case.block_tables.cuda(), case.context_lens.cuda(), case.q_start.cuda()
    out = torch.empty_like(q)
    ws = torch.zeros(b.pa_decode_multi_balanced_workspace_bytes(2, 2, 128), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(b.PagedKVError) as e:       # 9 tokens x 8 heads > 64 columns
        b.pa_decode_multi_balanced(q, k, v, bt, cl, qs, 9, case.scale, ws, out)
    assert e.value.status == -2
    b.pa_kv_append(case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda(), k, v)
    b.pa_decode_multi(q, k, v, bt, cl, qs, 9, case.scale, out)   # the row-block kernel
    torch.cuda.synchronize()
    P.assert_close(P.to_f64(out), oracle_multi(case), "max_q_len 9 on the row-block kernel")
    with pytest.raises(b.PagedKVError) as e:       # split mode without buffers
        b._check("pa_decode_multi", b._lib.pa_decode_multi(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), bt.data_ptr(), bt.shape[1], cl.data_ptr(),
            qs.data_ptr(), 2, case.rows, 3, 16, 2, 128, 16, case.num_blocks, case.scale, 16, 4,
            None, None, None, out.data_ptr(), None))
    assert e.value.status == -4


def test_rows_above_max_q_len_set_the_shape_bit(cuda_lib, multi_kernel):
    b = cuda_lib
    case = wl.make_multi_case("shape", 71, [20, 30], [1, 5], 8, 2, 128, 16)
    q, k, v = case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda()
    out = torch.zeros_like(q)
    b.pa_decode_multi(q, k, v, case.block_tables.cuda(), case.context_lens.cuda(),
                      case.q_start.cuda(), 4, case.scale, out)     # sequence 1 has 5 > 4
    torch.cuda.synchronize()
    assert b.pa_last_device_error() & 16
    assert b.pa_last_device_error() == 0           # read and cleared


def test_validating_mode_rejects_bad_q_start(cuda_lib):
    code = r"""
import torch
from paged_kv_cache_45_gb300 import binding as b, workloads as wl
case = wl.make_multi_case("val", 72, [20, 3], [4, 5], 8, 2, 128, 16)   # 5 rows, 8 tokens
q, k, v = case.q.cuda(), case.k_cache.cuda(), case.v_cache.cuda()
out = torch.empty_like(q)
bad = torch.tensor([0, 4, 10], dtype=torch.int32, device="cuda")      # ends past the rows
try:
    b.pa_decode_multi(q, k, v, case.block_tables.cuda(), case.context_lens.cuda(), bad, 8,
                      case.scale, out)
    print("accepted")
except b.PagedKVError as e:
    print("status", e.status)
"""
    env = dict(os.environ, PA_VALIDATE="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))), timeout=300)
    assert "status -1" in r.stdout, r.stdout + r.stderr
