"""Pins for the oracle's FP8 (e4m3) KV cache: the format's defining values,
exhaustive round trips and ties over the 256 codes, saturation, an independent
library conversion (torch.float8_e4m3fn), the quantization error bound, and
attention over a quantized pool against torch SDPA on the dequantized rows."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl


def test_format_defining_values():
    v = oracle.e4m3_value
    assert v(0x7E) == 448.0                  # largest finite
    assert v(0x08) == 2.0 ** -6              # smallest normal
    assert v(0x01) == 2.0 ** -9              # smallest subnormal
    assert v(0x38) == 1.0 and v(0xB8) == -1.0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    assert v(0x00) == 0.0 and v(0x80) == 0.0
    finite = [v(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(finite, finite[1:]))     # increasing magnitudes


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def test_midpoints_round_to_the_even_code():
    for c in range(0x7E):
        lo, hi = oracle.e4m3_value(c), oracle.e4m3_value(c + 1)
        mid = (lo + hi) / 2
        want = c if c % 2 == 0 else c + 1
        assert int(oracle.e4m3_encode([mid])[0]) == want, hex(c)
        assert int(oracle.e4m3_encode([-mid])[0]) == want | 0x80
        assert int(oracle.e4m3_encode([np.nextafter(mid, 0)])[0]) == c
        assert int(oracle.e4m3_encode([np.nextafter(mid, 1e9)])[0]) == c + 1


def test_saturates_and_keeps_nan():
    codes = oracle.e4m3_encode([449.0, 1e6, -1e6, math.inf, -math.inf, math.nan])
    assert list(codes) == [0x7E, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F]


def test_matches_torch_float8_e4m3fn_in_range():
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(20000, generator=g) * 40,
                   torch.randn(5000, generator=g) * 2.0 ** -7,       # subnormals
                   torch.rand(5000, generator=g) * 896 - 448])
    ours = oracle.e4m3_encode(x.numpy())
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_quantization_error_is_within_half_a_step():
    x = np.random.default_rng(1).normal(size=10000) * 30
    back = oracle.e4m3_decode(oracle.e4m3_encode(x))
    normal = np.abs(x) >= 2.0 ** -6
    rel = np.abs(back - x)[normal] / np.abs(x)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-12        # 3 mantissa bits: half ulp <= 2^-4


def test_quantize_rows_divides_in_float32_per_head():
    rows = wl.randn_bf16(torch.Generator().manual_seed(2), (5, 3, 16))
    scales = np.array([0.03, 0.05, 0.125], dtype=np.float32)
    got = oracle.quantize_rows_e4m3(wl.bits(rows), scales)
    ref = (rows.float() / torch.from_numpy(scales)[:, None]).to(torch.float8_e4m3fn)
    assert np.array_equal(got, ref.view(torch.uint8).numpy())


def test_fp8_decode_matches_sdpa_on_dequantized_rows():
    case = wl.make_case("fp8", 3, [1, 9, 40, 130], 8, 2, 64, 16, append=False)
    f8 = wl.fp8_pool(case, seed=3)
    kc, vc = f8["k_codes"].numpy(), f8["v_codes"].numpy()
    ks, vs = f8["k_scale"].numpy(), f8["v_scale"].numpy()
    got = pa.decode_fp8(wl.bits(case.q), kc, vc, ks, vs, case.block_tables.numpy(),
                        case.context_lens.numpy(), case.scale)
    K = torch.from_numpy(pa.dequantize_pool(kc, ks))
    V = torch.from_numpy(pa.dequantize_pool(vc, vs))
    q = torch.from_numpy(pa.bf16_bits_to_f64(wl.bits(case.q)))
    for b in range(case.batch):
        ctx = int(case.context_lens[b])
        t = torch.arange(ctx)
        blk = case.block_tables[b].long()[t // 16]
        Kb = K[blk, t % 16].permute(1, 0, 2).repeat_interleave(4, 0)
        Vb = V[blk, t % 16].permute(1, 0, 2).repeat_interleave(4, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q[b].unsqueeze(1), Kb, Vb,
                                                               scale=case.scale)[:, 0]
        np.testing.assert_allclose(got[b], ref.numpy(), rtol=0, atol=1e-12)


def test_fp8_append_writes_quantized_rows_at_slots():
    case = wl.make_case("fp8a", 4, [0, 5, 16, 31], 4, 2, 64, 16)
    f8 = wl.fp8_pool(case, seed=4)
    kc, vc = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    ks, vs = f8["k_scale"].numpy(), f8["v_scale"].numpy()
    pa.kv_append_fp8_inplace(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new),
                             case.slot_mapping.numpy(), ks, vs)
    for b in range(case.batch):
        s = int(case.slot_mapping[b])
        assert np.array_equal(kc[s // 16, s % 16], oracle.quantize_rows_e4m3(
            wl.bits(case.k_new)[b], ks))
    touched = np.zeros(kc.shape[:2], bool)
    for s in case.slot_mapping.tolist():
        touched[s // 16, s % 16] = True
    assert np.array_equal(kc[~touched], f8["k_codes"].numpy()[~touched])
