"""GPU parity on the two largest workloads, in the launch configuration the
bench times: the 70B-shape continuous batch (32 iterations of finish / join /
append / decode over a NaN-poisoned pool) and the 131072-token contexts split
into 4096-token ranges merged by the log-sum-exp reduce."""

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,iterations", [(0, 32), (1, 8)])
def test_continuous_batching_70b_shape(cuda_lib, seed, iterations):
    b = cuda_lib
    cb = wl.ContinuousBatching(seed=seed, iterations=iterations)
    kc_cpu, vc_cpu = cb.initial_caches("cpu")
    kc, vc = kc_cpu.cuda(), vc_cpu.cuda()
    kf, vf = kc_cpu.cuda(), vc_cpu.cuda()          # a second pool for the fused step
    ko, vo = wl.bits(kc_cpu), wl.bits(vc_cpu)          # oracle state (CPU, updated in place)
    rng = np.random.default_rng(seed)
    max_ctx = cb.max_blocks * cb.bs
    ws_bal = b.DecodeWorkspace(cb.B, cb.Hq, cb.D, b.BALANCED, device="cuda", num_kv_heads=cb.Hkv)
    fused_out = torch.empty((cb.B, cb.Hq, cb.D), dtype=torch.bfloat16, device="cuda")
    for it in range(cb.iterations):
        st = cb.step(it)
        for cache in (kc, vc, kf, vf):
            wl.poison_blocks(cache, st.freed)
        if st.freed:
            ko[st.freed] = wl.BF16_NAN_BITS
            vo[st.freed] = wl.BF16_NAN_BITS
        if st.fill_slots.numel():
            b.pa_kv_append(st.fill_k.cuda(), st.fill_v.cuda(), st.fill_slots.cuda(), kc, vc)
            b.pa_kv_append(st.fill_k.cuda(), st.fill_v.cuda(), st.fill_slots.cuda(), kf, vf)
            pa.kv_append_inplace(ko, vo, wl.bits(st.fill_k), wl.bits(st.fill_v),
                                 st.fill_slots.numpy())
        b.pa_kv_append(st.k_new.cuda(), st.v_new.cuda(), st.slot_mapping.cuda(), kc, vc)
        pa.kv_append_inplace(ko, vo, wl.bits(st.k_new), wl.bits(st.v_new),
                             st.slot_mapping.numpy())
        qd, btd, cld = st.q.cuda(), st.block_tables.cuda(), st.context_lens.cuda()
        # the bench's step: append fused into the balanced decode, one launch
        b.pa_append_decode(qd, st.k_new.cuda(), st.v_new.cuda(), st.slot_mapping.cuda(), kf, vf,
                           btd, cld, cb.scale, ws_bal.scratch, fused_out)
        got_fused = P.to_f64(fused_out)
        b.decode(qd, kc, vc, btd, cld, cb.scale, ws=ws_bal)            # separate launches
        got = P.to_f64(ws_bal.out)
        split = b.plan_split(st.context_lens.numpy(), cb.Hkv, b.num_sms())
        out_split = b.decode(qd, kc, vc, btd, cld, cb.scale, split_tokens=split,
                             max_context=max_ctx)
        got_split = P.to_f64(out_split)
        assert np.isfinite(got).all(), f"iteration {it}: NaN leaked from a poisoned block"
        assert np.isfinite(got_fused).all(), f"iteration {it}: NaN leaked (fused step)"
        assert np.isfinite(got_split).all(), f"iteration {it}: NaN leaked (split {split})"
        if it in (0, cb.iterations - 1):
            seqs = np.arange(cb.B)
        else:
            joiners = [j for j, _ in cb.schedule[it]["joins"]]
            longest = [int(np.argmax(st.context_lens.numpy()))]
            seqs = np.unique(np.concatenate([rng.choice(cb.B, 12, replace=False), joiners,
                                             longest]).astype(int))
        ref = pa.decode(wl.bits(st.q), ko, vo, st.block_tables.numpy(), st.context_lens.numpy(),
                        cb.scale, seqs=seqs)
        P.assert_close(got_fused[seqs], ref, f"iteration {it} fused step")
        P.assert_close(got[seqs], ref, f"iteration {it} balanced")
        P.assert_close(got_split[seqs], ref, f"iteration {it} split={split}")
    torch.cuda.synchronize()
    # the whole pool after 32 iterations of appends, fills and poisoning: bit-exact
    assert np.array_equal(wl.bits(kc.cpu()), ko)
    assert np.array_equal(wl.bits(vc.cpu()), vo)
    assert np.array_equal(wl.bits(kf.cpu()), ko)
    assert np.array_equal(wl.bits(vf.cpu()), vo)
    assert b.pa_last_device_error() == 0


@pytest.mark.parametrize("split", [4096, "planned", -1])
def test_long_context_split_reduce(cuda_lib, split):
    case = wl.long_context_case(0)
    if split == "planned":
        split = cuda_lib.plan_split(case.context_lens.numpy(), 8, cuda_lib.num_sms())
    d = P.dev(case)
    out = cuda_lib.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                          case.scale, split_tokens=split, max_context=131072)
    got = P.to_f64(out)
    ref = P.oracle_out(case)
    P.assert_close(got, ref, f"131072 tokens split={split}")
