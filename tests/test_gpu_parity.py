"""GPU parity: the sm_103a kernels, called through the C ABI, against the fp64
oracle on the same seeded inputs.

* pa_kv_append and all block indexing: bit-exact.
* pa_decode (+ pa_decode_splitk_reduce): max abs error <= 2e-2 and per-row
  relative L2 <= 5e-3 against the oracle (tests/parity.py).
Sizes span several 16-token tiles, every block size, ragged tails, empty
contexts and empty splits.
"""

import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


def run_step(b, case, split=0, max_context=None):
    """Append (if any) then decode on the GPU; returns (out, k_cache, v_cache)."""
    d = P.dev(case)
    if case.k_new is not None:
        b.pa_kv_append(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    out = b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   case.scale, split_tokens=split, max_context=max_context)
    torch.cuda.synchronize()
    return out, d["k_cache"], d["v_cache"]


# ---------------------------------------------------------------------------
# append: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("maker", [lambda: wl.tiny_case(0),
                                   lambda: wl.make_case("s", 1, [0, 1, 15, 16, 31, 32, 33, 200],
                                                        8, 2, 64, 8),
                                   lambda: wl.llama8b_case(0, batch=64)],
                         ids=["tiny", "ragged_bs8", "8b_full"])
def test_append_bit_exact(cuda_lib, maker):
    case = maker()
    d = P.dev(case)
    cuda_lib.pa_kv_append(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    torch.cuda.synchronize()
    kc, vc = P.oracle_caches(case)
    assert np.array_equal(wl.bits(d["k_cache"].cpu()), kc)
    assert np.array_equal(wl.bits(d["v_cache"].cpu()), vc)


def test_append_skips_negative_and_out_of_pool_slots(cuda_lib):
    case = wl.make_case("s", 2, [3, 4, 5, 6], 2, 1, 64, 16)
    d = P.dev(case)
    before_k = d["k_cache"].clone()
    nslots = case.num_blocks * case.block_size
    slots = torch.tensor([-1, nslots, nslots + 100, -7], dtype=torch.int64, device="cuda")
    cuda_lib.pa_kv_append(d["k_new"], d["v_new"], slots, d["k_cache"], d["v_cache"])
    torch.cuda.synchronize()
    assert torch.equal(before_k.view(torch.int16), d["k_cache"].view(torch.int16))


def test_append_many_rows_prefill_style(cuda_lib):
    # a joiner's whole prompt written through the same entry point
    case = wl.make_case("p", 3, [0, 0], 8, 8, 128, 16, append=False, num_blocks=40)
    g = torch.Generator().manual_seed(5)
    T = 300
    rows = torch.randn((T, 8, 128), generator=g).to(torch.bfloat16)
    rows_v = torch.randn((T, 8, 128), generator=g).to(torch.bfloat16)
    slots = torch.from_numpy(np.random.default_rng(1).permutation(40 * 16)[:T].astype(np.int64))
    d = P.dev(case)
    cuda_lib.pa_kv_append(rows.cuda(), rows_v.cuda(), slots.cuda(), d["k_cache"], d["v_cache"])
    torch.cuda.synchronize()
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(rows),
                          wl.bits(rows_v), slots.numpy())
    assert np.array_equal(wl.bits(d["k_cache"].cpu()), kc)
    assert np.array_equal(wl.bits(d["v_cache"].cpu()), vc)


# ---------------------------------------------------------------------------
# decode: against the oracle
# ---------------------------------------------------------------------------

def test_tiny_case(cuda_lib):
    case = wl.tiny_case(0)
    for split in (0, 16, BAL):
        out, _, _ = run_step(cuda_lib, case, split=split)
        P.assert_close(P.to_f64(out), P.oracle_out(case), f"tiny split={split}")


LENS = [0, 1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 1000]
BAL = -1  # binding.BALANCED: the work-balanced persistent schedule


@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (6, 2), (16, 2)])
def test_group_and_head_dim_sweep(cuda_lib, d, hq, hkv, sched):
    case = wl.make_case("sweep", 100 + d + hq * 3 + hkv, LENS, hq, hkv, d, 16)
    out, _, _ = run_step(cuda_lib, case, split=sched)
    P.assert_close(P.to_f64(out), P.oracle_out(case), f"G={hq // hkv} D={d} sched={sched}")


@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32, 64, 256])
def test_every_block_size(cuda_lib, bs, sched):
    case = wl.make_case("bs", 200 + bs, LENS, 8, 2, 128, bs)
    out, _, _ = run_step(cuda_lib, case, split=sched)
    P.assert_close(P.to_f64(out), P.oracle_out(case), f"bs={bs} sched={sched}")


@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_every_short_context(cuda_lib, g, d, sched):
    # the tiny-shape sweep: every context length 1..40 (40 sequences, one
    # appended token each) for each block size 1, 8, 16, 32
    for bs in (1, 8, 16, 32):
        case = wl.make_case("short", 900 + 10 * g + d + bs, list(range(40)), 2 * g, 2, d, bs)
        out, _, _ = run_step(cuda_lib, case, split=sched)
        P.assert_close(P.to_f64(out), P.oracle_out(case), f"G={g} D={d} bs={bs} sched={sched}")


@pytest.mark.parametrize("lens", [[5], [0, 0, 3], [1] * 7, [2000, 1, 0, 17, 4096, 33] * 20,
                                  list(range(0, 700, 7))],
                         ids=["one_seq", "mostly_empty", "fewer_tiles_than_workers", "mixed_120",
                              "ramp_100"])
def test_balanced_partitions(cuda_lib, lens):
    # fewer tiles than workers, units cut by many workers, empty sequences
    case = wl.make_case("bal", 600 + len(lens), lens, 8, 2, 128, 16)
    out, _, _ = run_step(cuda_lib, case, split=BAL)
    P.assert_close(P.to_f64(out), P.oracle_out(case), f"balanced {len(lens)} seqs")


def test_balanced_workspace_is_reusable_and_deterministic(cuda_lib):
    b = cuda_lib
    case = wl.make_case("bal_ws", 610, [3000, 5, 800, 0, 1234, 64] * 8, 8, 2, 128, 16,
                        append=False)
    d = P.dev(case)
    ws = b.DecodeWorkspace(case.batch, 8, 128, b.BALANCED, device="cuda", num_kv_heads=2)
    outs = []
    for _ in range(3):
        b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                 case.scale, ws=ws)
        outs.append(ws.out.clone())
    torch.cuda.synchronize()
    counters = ws.scratch[: case.batch * 2 * 4].view(torch.int32)
    assert torch.all(counters == 0), "counters not left at zero"
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
    P.assert_close(P.to_f64(outs[0]), P.oracle_out(case), "balanced reuse")


def test_batch_size_may_shrink_and_grow_between_calls(cuda_lib):
    # the kernel's shared memory grows with the batch (its prefix sums); a
    # smaller batch in between must not leave the kernel unable to launch the
    # larger one again
    rng = np.random.default_rng(5)
    big = wl.make_case("grow", 620, list(rng.integers(1, 40, 2999)), 8, 2, 128, 16)
    small = wl.make_case("shrink", 621, [5, 70, 300] * 4 + [9], 8, 2, 128, 16)
    for case in (big, small, big, small):
        out, _, _ = run_step(cuda_lib, case, split=BAL)
        seqs = None if case.batch < 100 else list(range(0, case.batch, 37))
        got = P.to_f64(out) if seqs is None else P.to_f64(out)[seqs]
        P.assert_close(got, P.oracle_out(case, seqs=seqs), f"B={case.batch}")


def test_largest_batches(cuda_lib):
    # The balanced kernel keeps the batch's tile prefix sums in shared memory:
    # 30,000 sequences still fit (one block per SM); 60,000 do not and are
    # refused with PA_ERR_UNSUPPORTED before any launch, while the fixed-split
    # kernel (one block per sequence x KV head, grid z up to 65,535) runs them.
    b = cuda_lib
    rng = np.random.default_rng(9)
    for B in (30000, 60000):
        case = wl.make_case(f"big{B}", 630, list(rng.integers(0, 4, B)), 8, 2, 128, 16,
                            append=False)
        d = P.dev(case)
        seqs = list(range(0, B, 997)) + [B - 1]
        want = P.oracle_out(case, seqs=seqs)
        if B == 30000:
            out = b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                           d["context_lens"], case.scale, split_tokens=b.BALANCED)
            torch.cuda.synchronize()
            P.assert_close(P.to_f64(out)[seqs], want, "balanced B=30000")
        else:
            with pytest.raises(b.PagedKVError) as e:
                b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                         d["context_lens"], case.scale, split_tokens=b.BALANCED)
            assert e.value.status == -2
            out = b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                           d["context_lens"], case.scale)
            torch.cuda.synchronize()
            P.assert_close(P.to_f64(out)[seqs], want, "fixed split B=60000")
        assert b.pa_last_device_error() == 0


def test_balanced_rejects_small_workspace(cuda_lib):
    b = cuda_lib
    case = wl.tiny_case(0)
    d = P.dev(case)
    need = b.pa_decode_balanced_workspace_bytes(case.batch, 1, 64)
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    with pytest.raises(b.PagedKVError) as e:
        b.pa_decode_balanced(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], case.scale, small, out)
    assert e.value.status == -4


@pytest.mark.parametrize("split", [16, 32, 256, 4096])
def test_context_splits_and_reduce(cuda_lib, split):
    case = wl.make_case("split", 300, LENS + [2049, 4000], 8, 2, 128, 16)
    out, _, _ = run_step(cuda_lib, case, split=split)
    P.assert_close(P.to_f64(out), P.oracle_out(case), f"split={split}")


def test_split_partials_match_oracle_partials(cuda_lib):
    case = wl.make_case("part", 301, [0, 5, 40, 300], 8, 2, 64, 16, append=False)
    split, S = 32, 12
    d = P.dev(case)
    po = torch.full((4, 8, S, 64), float("nan"), device="cuda")
    pl = torch.full((4, 8, S), float("nan"), device="cuda")
    out = torch.empty((4, 8, 64), dtype=torch.bfloat16, device="cuda")
    cuda_lib.pa_decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                       case.scale, out, split, S, po, pl)
    torch.cuda.synchronize()
    ref_o, ref_l = pa.decode_split_partials(wl.bits(case.q), wl.bits(case.k_cache),
                                            wl.bits(case.v_cache), case.block_tables.numpy(),
                                            case.context_lens.numpy(), case.scale, split, S)
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    for b, ctx in enumerate(case.context_lens.tolist()):
        n = -(-ctx // split)
        if n:
            np.testing.assert_allclose(pl[b, :, :n], ref_l[b, :, :n], rtol=0, atol=2e-3)
            np.testing.assert_allclose(po[b, :, :n], ref_o[b, :, :n], rtol=0, atol=1e-2)
        assert np.isnan(pl[b, :, n:]).all()      # splits past the context are not written


@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
def test_context_of_one_returns_v_exactly(cuda_lib, sched):
    case = wl.make_case("one", 400, [0, 0, 0], 8, 1, 128, 16)   # append 1 -> ctx 1
    out, _, _ = run_step(cuda_lib, case, split=sched)
    v = case.v_new.float()                                          # [B, 1, D]
    assert torch.equal(out.float().cpu(), v.expand(-1, 8, -1))


def test_identical_keys_give_mean_of_v(cuda_lib):
    case = wl.make_case("same", 401, [300, 47], 4, 1, 128, 16, append=False)
    kf = case.k_cache.view(-1, 1, 128)
    for b, blocks in enumerate(case.seq_blocks):
        rows = torch.from_numpy(wl.token_rows(blocks, int(case.context_lens[b]), 16))
        kf[rows] = kf[rows[0]].clone()
    out, _, _ = run_step(cuda_lib, case)
    ref = P.oracle_out(case)
    for b, blocks in enumerate(case.seq_blocks):
        V = pa.bf16_bits_to_f64(pa.gather_sequence(wl.bits(case.v_cache), case.block_tables[b].numpy(),
                                                   int(case.context_lens[b])))
        np.testing.assert_allclose(ref[b, 0], V[:, 0].mean(0), atol=1e-12)
    P.assert_close(P.to_f64(out), ref, "identical keys")


def test_empty_contexts_give_zero_rows(cuda_lib):
    case = wl.make_case("empty", 402, [0, 0, 50], 8, 2, 128, 16, append=False)
    for split in (0, 32, BAL):
        out, _, _ = run_step(cuda_lib, case, split=split, max_context=64)
        o = out.float().cpu()
        assert torch.all(o[:2] == 0) and torch.isfinite(o).all()
        P.assert_close(P.to_f64(out), P.oracle_out(case), f"empty split={split}")


# ---------------------------------------------------------------------------
# invariances on the GPU (block ids are names only)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
def test_gpu_block_permutation_is_bit_invisible(cuda_lib, sched):
    case = wl.make_case("perm", 500, LENS, 8, 2, 128, 16)
    out1, _, _ = run_step(cuda_lib, case, split=sched)
    rng = np.random.default_rng(3)
    pi = np.concatenate([[0], 1 + rng.permutation(case.num_blocks - 1)])
    pit = torch.from_numpy(pi)
    perm = wl.DecodeCase(**{**case.__dict__})
    perm.k_cache = torch.empty_like(case.k_cache); perm.k_cache[pit] = case.k_cache
    perm.v_cache = torch.empty_like(case.v_cache); perm.v_cache[pit] = case.v_cache
    perm.block_tables = torch.from_numpy(pi[case.block_tables.numpy()].astype(np.int32))
    s = case.slot_mapping.numpy()
    perm.slot_mapping = torch.from_numpy(pi[s // 16] * 16 + s % 16)
    out2, _, _ = run_step(cuda_lib, perm, split=sched)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def copied_prefix_case(case, prefix_blocks):
    """The case with every sequence but the first reading its own copy of the
    shared prefix blocks (appended after the pool), the same rows otherwise."""
    bt = case.block_tables.numpy()
    assert (bt[:, :prefix_blocks] == bt[0, :prefix_blocks]).all()
    B, nb = bt.shape[0], case.num_blocks
    src = torch.from_numpy(np.tile(bt[0, :prefix_blocks], B - 1).astype(np.int64))
    bt2 = bt.copy()
    for i in range(1, B):
        bt2[i, :prefix_blocks] = nb + (i - 1) * prefix_blocks + np.arange(prefix_blocks)
    cp = wl.DecodeCase(**{**case.__dict__})
    cp.k_cache = torch.cat([case.k_cache, case.k_cache[src]])
    cp.v_cache = torch.cat([case.v_cache, case.v_cache[src]])
    cp.block_tables = torch.from_numpy(bt2)
    cp.num_blocks = nb + (B - 1) * prefix_blocks
    return cp


@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
def test_gpu_shared_prefix_equals_copied_prefix(cuda_lib, sched):
    # sharing is only naming: the same rows reached through one set of
    # prefix blocks or through private copies give the same bits
    pref = 256
    case = wl.make_case("pfxg", 510, [pref + x for x in (0, 5, 16, 100, 700, 1)], 8, 2, 128, 16,
                        shared_prefix=pref)
    out1, _, _ = run_step(cuda_lib, case, split=sched)
    out2, _, _ = run_step(cuda_lib, copied_prefix_case(case, pref // 16), split=sched)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    P.assert_close(P.to_f64(out1), P.oracle_out(case), f"shared prefix sched={sched}")


@pytest.mark.parametrize("sched", [0, BAL], ids=["per_split", "balanced"])
def test_gpu_block_size_1_vs_16_bit_identical(cuda_lib, sched):
    lens = [5, 16, 40, 129]
    c16 = wl.make_case("b16", 501, lens, 8, 2, 128, 16, append=False)
    kc, vc = wl.bits(c16.k_cache), wl.bits(c16.v_cache)
    bt, cl = c16.block_tables.numpy(), c16.context_lens.numpy()
    nb1 = int(cl.sum()) + 1
    k1 = np.full((nb1, 1, 2, 128), wl.BF16_NAN_BITS, np.uint16)
    v1 = k1.copy()
    tab1 = np.zeros((4, int(cl.max())), np.int32)
    nxt = 1
    for b in range(4):
        K = pa.gather_sequence(kc, bt[b], int(cl[b]))
        V = pa.gather_sequence(vc, bt[b], int(cl[b]))
        for t in range(int(cl[b])):
            tab1[b, t] = nxt
            k1[nxt, 0], v1[nxt, 0] = K[t], V[t]
            nxt += 1
    c1 = wl.DecodeCase(**{**c16.__dict__})
    c1.block_size, c1.num_blocks = 1, nb1
    c1.k_cache = torch.from_numpy(k1.view(np.int16)).view(torch.bfloat16)
    c1.v_cache = torch.from_numpy(v1.view(np.int16)).view(torch.bfloat16)
    c1.block_tables = torch.from_numpy(tab1)
    o16, _, _ = run_step(cuda_lib, c16, split=sched)
    o1, _, _ = run_step(cuda_lib, c1, split=sched)
    assert torch.equal(o16.view(torch.int16), o1.view(torch.int16))


# ---------------------------------------------------------------------------
# the full-size 8B and prefix-sharing workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_8b_workload_full(cuda_lib, seed):
    case = wl.llama8b_case(seed)
    split = cuda_lib.plan_split(case.context_lens.numpy(), 8, cuda_lib.num_sms())
    out, _, _ = run_step(cuda_lib, case, split=split,
                         max_context=int(case.context_lens.max()))
    P.assert_close(P.to_f64(out), P.oracle_out(case), f"8b seed={seed} split={split}")
    ref = P.oracle_out(case)
    for sched in (0, BAL):
        o, _, _ = run_step(cuda_lib, case, split=sched)
        P.assert_close(P.to_f64(o), ref, f"8b seed={seed} sched={sched}")


def test_prefix_sharing_full(cuda_lib):
    case = wl.prefix_sharing_case(0)
    split = cuda_lib.plan_split(case.context_lens.numpy(), 8, cuda_lib.num_sms())
    out, _, _ = run_step(cuda_lib, case, split=split, max_context=int(case.context_lens.max()))
    ref = P.oracle_out(case)
    P.assert_close(P.to_f64(out), ref, f"prefix split={split}")
    out, _, _ = run_step(cuda_lib, case, split=BAL)
    P.assert_close(P.to_f64(out), ref, "prefix balanced")


def test_device_error_word_is_clear(cuda_lib):
    run_step(cuda_lib, wl.tiny_case(0))
    assert cuda_lib.pa_last_device_error() == 0


def test_validating_mode_rejects_bad_tables(cuda_lib):
    code = r"""
import torch, sys
sys.path.insert(0, %r)
from paged_kv_cache_45_gb300 import binding as b, workloads as wl
c = wl.tiny_case(0)
q, kc, vc = c.q.cuda(), c.k_cache.cuda(), c.v_cache.cuda()
bt, cl = c.block_tables.clone(), c.context_lens.cuda()
out = torch.empty_like(q)
b.pa_decode(q, kc, vc, bt.cuda(), cl, c.scale, out)
bad = bt.clone(); bad[3, 1] = c.num_blocks
try:
    b.pa_decode(q, kc, vc, bad.cuda(), cl, c.scale, out)
    print("accepted")
except b.PagedKVError as e:
    print("rejected", e.status)
""" % os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PA_VALIDATE="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert "rejected -1" in r.stdout


FMA_SCRIPT = r"""
import sys, torch, numpy as np
sys.path.insert(0, %r)
from paged_kv_cache_45_gb300 import binding as b, workloads as wl
from oracle import paged_attention as pa
from tests import parity as P
cases = [wl.tiny_case(0),
         wl.make_case("fma", 800, [0, 1, 15, 16, 17, 33, 100, 1000, 3000], 8, 1, 128, 16),
         wl.make_case("fma64", 801, [5, 40, 600], 8, 2, 64, 16),
         wl.make_case("fma_bs1", 802, [20, 70], 4, 1, 128, 1)]
for c in cases:
    d = P.dev(c)
    b.pa_kv_append(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    out = b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   c.scale, split_tokens=b.BALANCED)
    torch.cuda.synchronize()
    P.assert_close(P.to_f64(out), P.oracle_out(c), c.name)
print("fma ok")
"""


def test_fma_ablation_matches_oracle(cuda_lib):
    # the CUDA-core ablation of the tile math (PA_DECODE_MATH=fma, read once
    # per process) must compute the same attention
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PA_DECODE_MATH="fma")
    r = subprocess.run([sys.executable, "-c", FMA_SCRIPT % root], env=env, capture_output=True,
                       text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "fma ok" in r.stdout


@pytest.mark.parametrize("lens,hq,hkv,d,bs", [
    ([1, 7, 16, 33], 2, 1, 64, 16),                           # the tiny workload
    (LENS, 8, 2, 128, 16),
    ([0, 15, 16, 31, 47, 300, 1023, 2048], 8, 1, 128, 8),
    ([3, 40, 600, 17], 4, 4, 64, 1),
    ([5000, 2, 9, 128] * 12, 16, 2, 128, 32),
], ids=["tiny", "edges", "bs8_g8", "bs1_mha", "mixed_bs32"])
def test_fused_append_decode_matches_append_then_decode(cuda_lib, lens, hq, hkv, d, bs):
    b = cuda_lib
    case = wl.make_case("fused", 900 + len(lens) + bs, lens, hq, hkv, d, bs)
    dv = P.dev(case)
    ws = torch.zeros(b.pa_decode_balanced_workspace_bytes(case.batch, hkv, d), dtype=torch.uint8,
                     device="cuda")
    out = torch.full_like(dv["q"], float("nan"))
    b.pa_append_decode(dv["q"], dv["k_new"], dv["v_new"], dv["slot_mapping"], dv["k_cache"],
                       dv["v_cache"], dv["block_tables"], dv["context_lens"], case.scale, ws, out)
    torch.cuda.synchronize()
    kc, vc = P.oracle_caches(case)
    assert np.array_equal(wl.bits(dv["k_cache"].cpu()), kc)     # the append, bit-exact
    assert np.array_equal(wl.bits(dv["v_cache"].cpu()), vc)
    P.assert_close(P.to_f64(out), P.oracle_out(case, caches=(kc, vc)), "fused step")


def test_fused_append_skips_negative_slots(cuda_lib):
    b = cuda_lib
    case = wl.make_case("fused_skip", 950, [20, 33, 7], 8, 2, 128, 16)
    dv = P.dev(case)
    slots = dv["slot_mapping"].clone()
    slots[1] = -1
    ws = torch.zeros(b.pa_decode_balanced_workspace_bytes(3, 2, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(dv["q"])
    b.pa_append_decode(dv["q"], dv["k_new"], dv["v_new"], slots, dv["k_cache"], dv["v_cache"],
                       dv["block_tables"], dv["context_lens"], case.scale, ws, out)
    torch.cuda.synchronize()
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), slots.cpu().numpy())
    assert np.array_equal(wl.bits(dv["k_cache"].cpu()), kc)
    o = P.to_f64(out)
    ref = P.oracle_out(case, caches=(kc, vc))
    # sequence 1 attends over its (NaN-poisoned) unwritten slot, like append-then-decode
    assert np.isnan(ref[1]).all()
    P.assert_close(o[[0, 2]], ref[[0, 2]], "fused step with a skipped slot")
