"""GPU parity for the FP8 (e4m3) KV cache against the fp64 oracle.

* pa_kv_append_fp8 and the fused append: the codes, bit-exact (both sides
  divide by the head's scale in fp32 and round to the nearest even code).
* pa_decode_balanced_fp8 / pa_append_decode_fp8: the parity bar of the bf16
  path (max abs <= 2e-2, per-row relative L2 <= 5e-3) against attention over
  the dequantized pool.
"""

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

FP8_NAN = 0x7F


def fp8_dev(case, seed):
    f8 = wl.fp8_pool(case, seed)
    d = P.dev(case)
    d.update(k_codes=f8["k_codes"].cuda(), v_codes=f8["v_codes"].cuda(),
             k_scale=f8["k_scale"].cuda(), v_scale=f8["v_scale"].cuda())
    return f8, d


def oracle_after_append(case, f8, slots=None):
    kc, vc = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    if case.k_new is not None:
        s = case.slot_mapping.numpy() if slots is None else slots
        pa.kv_append_fp8_inplace(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new), s,
                                 f8["k_scale"].numpy(), f8["v_scale"].numpy())
    return kc, vc


def oracle_decode(case, f8, kc, vc, seqs=None):
    return pa.decode_fp8(wl.bits(case.q), kc, vc, f8["k_scale"].numpy(), f8["v_scale"].numpy(),
                         case.block_tables.numpy(), case.context_lens.numpy(), case.scale, seqs)


def workspace(b, case):
    return torch.zeros(b.pa_decode_balanced_workspace_bytes(case.batch, case.num_kv_heads,
                                                            case.head_dim),
                       dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("mul", [1.0, 2.0 ** -12, 500.0], ids=["normal", "subnormal", "saturate"])
def test_fp8_append_codes_bit_exact(cuda_lib, mul):
    b = cuda_lib
    case = wl.make_case("f8app", 10, [0, 3, 16, 31, 200], 8, 8, 128, 16)
    case.k_new = (case.k_new.float() * mul).to(torch.bfloat16)
    case.v_new = (case.v_new.float() * mul).to(torch.bfloat16)
    f8, d = fp8_dev(case, 10)
    b.pa_kv_append_fp8(case.k_new.cuda(), case.v_new.cuda(), d["slot_mapping"], d["k_codes"],
                       d["v_codes"], d["k_scale"], d["v_scale"])
    torch.cuda.synchronize()
    kc, vc = oracle_after_append(case, f8)
    assert np.array_equal(d["k_codes"].cpu().numpy(), kc)
    assert np.array_equal(d["v_codes"].cpu().numpy(), vc)


LENS = [0, 1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 1000]


@pytest.mark.parametrize("hq,hkv,bs", [(8, 8, 16), (8, 4, 16), (8, 2, 16), (8, 1, 16),
                                       (16, 2, 16), (8, 2, 1), (8, 2, 8), (8, 2, 32)])
def test_fp8_decode_matches_oracle(cuda_lib, hq, hkv, bs):
    b = cuda_lib
    case = wl.make_case("f8dec", 20 + hq + hkv + bs, LENS, hq, hkv, 128, bs, append=False)
    f8, d = fp8_dev(case, 20)
    out = torch.empty_like(d["q"])
    b.pa_decode_balanced_fp8(d["q"], d["k_codes"], d["v_codes"], d["k_scale"], d["v_scale"],
                             d["block_tables"], d["context_lens"], case.scale, workspace(b, case),
                             out)
    torch.cuda.synchronize()
    kc, vc = f8["k_codes"].numpy(), f8["v_codes"].numpy()
    P.assert_close(P.to_f64(out), oracle_decode(case, f8, kc, vc), f"fp8 G={hq // hkv} bs={bs}")


@pytest.mark.parametrize("lens,hq,hkv,bs", [([1, 7, 16, 33], 8, 2, 16),
                                            ([0, 40, 600, 4097, 17] * 8, 16, 2, 16),
                                            ([3, 40, 600], 8, 8, 1)],
                         ids=["small", "mixed", "bs1"])
def test_fp8_fused_step_matches_append_then_decode(cuda_lib, lens, hq, hkv, bs):
    b = cuda_lib
    case = wl.make_case("f8fused", 30 + len(lens), lens, hq, hkv, 128, bs)
    f8, d = fp8_dev(case, 30)
    out = torch.full_like(d["q"], float("nan"))
    b.pa_append_decode_fp8(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_codes"],
                           d["v_codes"], d["k_scale"], d["v_scale"], d["block_tables"],
                           d["context_lens"], case.scale, workspace(b, case), out)
    torch.cuda.synchronize()
    kc, vc = oracle_after_append(case, f8)
    assert np.array_equal(d["k_codes"].cpu().numpy(), kc)
    assert np.array_equal(d["v_codes"].cpu().numpy(), vc)
    P.assert_close(P.to_f64(out), oracle_decode(case, f8, kc, vc), "fp8 fused step")


def test_fp8_context_of_one_returns_dequantized_v(cuda_lib):
    b = cuda_lib
    case = wl.make_case("f8one", 40, [0, 0], 8, 2, 128, 16)
    f8, d = fp8_dev(case, 40)
    out = torch.empty_like(d["q"])
    b.pa_append_decode_fp8(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_codes"],
                           d["v_codes"], d["k_scale"], d["v_scale"], d["block_tables"],
                           d["context_lens"], case.scale, workspace(b, case), out)
    torch.cuda.synchronize()
    vq = pa.quantize_rows_e4m3(wl.bits(case.v_new), f8["v_scale"].numpy())   # [B, Hkv, D]
    v = pa.e4m3_decode(vq) * f8["v_scale"].numpy().astype(np.float64)[:, None]
    want = torch.from_numpy(v).float().to(torch.bfloat16).float().numpy()  # bf16 of code*scale
    got = out.float().cpu().numpy()
    for h in range(8):
        np.testing.assert_allclose(got[:, h], want[:, h // 4], rtol=0, atol=1e-2)


def test_fp8_continuous_batching_70b_shape(cuda_lib):
    b = cuda_lib
    cb = wl.ContinuousBatching(seed=1, iterations=12)
    kc_cpu, vc_cpu = cb.initial_caches("cpu")
    holder = wl.DecodeCase("cb", cb.Hq, cb.Hkv, cb.D, cb.bs, cb.num_blocks, cb.scale,
                           q=torch.zeros(1, cb.Hq, cb.D, dtype=torch.bfloat16), k_cache=kc_cpu,
                           v_cache=vc_cpu, block_tables=torch.zeros(1, 1, dtype=torch.int32),
                           context_lens=torch.zeros(1, dtype=torch.int32))
    f8 = wl.fp8_pool(holder, seed=5)
    del kc_cpu, vc_cpu
    ko, vo = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    kd, vd = f8["k_codes"].cuda(), f8["v_codes"].cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    ksn, vsn = f8["k_scale"].numpy(), f8["v_scale"].numpy()
    ws = torch.zeros(b.pa_decode_balanced_workspace_bytes(cb.B, cb.Hkv, cb.D), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((cb.B, cb.Hq, cb.D), dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(1)
    for it in range(cb.iterations):
        st = cb.step(it)
        if st.freed:
            idx = torch.as_tensor(st.freed, dtype=torch.long)
            kd[idx.cuda()] = FP8_NAN
            vd[idx.cuda()] = FP8_NAN
            ko[st.freed] = FP8_NAN
            vo[st.freed] = FP8_NAN
        if st.fill_slots.numel():
            b.pa_kv_append_fp8(st.fill_k.cuda(), st.fill_v.cuda(), st.fill_slots.cuda(), kd, vd,
                               ks, vs)
            pa.kv_append_fp8_inplace(ko, vo, wl.bits(st.fill_k), wl.bits(st.fill_v),
                                     st.fill_slots.numpy(), ksn, vsn)
        b.pa_append_decode_fp8(st.q.cuda(), st.k_new.cuda(), st.v_new.cuda(),
                               st.slot_mapping.cuda(), kd, vd, ks, vs, st.block_tables.cuda(),
                               st.context_lens.cuda(), cb.scale, ws, out)
        pa.kv_append_fp8_inplace(ko, vo, wl.bits(st.k_new), wl.bits(st.v_new),
                                 st.slot_mapping.numpy(), ksn, vsn)
        got = P.to_f64(out)
        assert np.isfinite(got).all(), f"iteration {it}: NaN leaked"
        seqs = np.unique(np.concatenate([rng.choice(cb.B, 10, replace=False),
                                         [int(np.argmax(st.context_lens.numpy()))]]))
        ref = pa.decode_fp8(wl.bits(st.q), ko, vo, ksn, vsn, st.block_tables.numpy(),
                            st.context_lens.numpy(), cb.scale, seqs=seqs)
        P.assert_close(got[seqs], ref, f"fp8 iteration {it}")
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), ko)
    assert np.array_equal(vd.cpu().numpy(), vo)
    assert b.pa_last_device_error() == 0
