"""Pins for the oracle's multi-token causal attention over an e4m3 pool
(oracle.decode_multi_fp8): one-token rows equal the e4m3 decode; over codes
whose read-back values are exact bf16 numbers it equals the bf16 multi-token
attention; a prompt processed in chunks equals full causal attention by torch
SDPA (fp64) on the dequantized rows; and swapped K/V scales are rejected."""

import numpy as np
import torch

import oracle
from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl


def quantized(case, k_scale, v_scale):
    """e4m3 codes of the case's pool after its append (unowned slots NaN)."""
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), case.slot_mapping.numpy())
    nb, bs, h, d = kc.shape
    kq = oracle.quantize_rows_e4m3(kc.reshape(-1, h, d), k_scale).reshape(kc.shape)
    vq = oracle.quantize_rows_e4m3(vc.reshape(-1, h, d), v_scale).reshape(vc.shape)
    return kq, vq


def test_one_token_rows_equal_the_e4m3_decode():
    case = wl.make_multi_case("f1", 1, [0, 3, 16, 40, 100], [1] * 5, 8, 2, 128, 16)
    ks, vs = np.array([0.03, 0.05]), np.array([0.04, 0.02])
    kq, vq = quantized(case, ks, vs)
    got = oracle.decode_multi_fp8(wl.bits(case.q), kq, vq, ks, vs, case.block_tables.numpy(),
                                  case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    want = oracle.decode_fp8(wl.bits(case.q), kq, vq, ks, vs, case.block_tables.numpy(),
                             case.context_lens.numpy(), case.scale)
    assert np.abs(got - want).max() < 1e-12


def test_exact_bf16_values_equal_the_bf16_multi_token_attention():
    # power-of-two scales: every read-back value (4 significant bits times
    # 2^k) is a bf16 number, so a bf16 pool can hold the same values
    case = wl.make_multi_case("f2", 2, [5, 0, 33, 64], [4, 3, 8, 1], 8, 2, 128, 16)
    ks, vs = np.array([2.0 ** -5, 2.0 ** -4]), np.array([2.0 ** -6, 2.0 ** -5])
    kq, vq = quantized(case, ks, vs)
    kf = pa.dequantize_pool(kq, ks).astype(np.float32)
    vf = pa.dequantize_pool(vq, vs).astype(np.float32)
    kb = (kf.view(np.uint32) >> 16).astype(np.uint16)       # exact: low half is zero
    vb = (vf.view(np.uint32) >> 16).astype(np.uint16)
    finite = np.isfinite(kf)
    assert np.all((kf.view(np.uint32)[finite] & 0xFFFF) == 0)
    got = oracle.decode_multi_fp8(wl.bits(case.q), kq, vq, ks, vs, case.block_tables.numpy(),
                                  case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    want = oracle.decode_multi(wl.bits(case.q), kb, vb, case.block_tables.numpy(),
                               case.context_lens.numpy(), case.q_start.numpy(), case.scale)
    assert np.abs(got - want).max() < 1e-12


def test_chunked_prompt_equals_full_causal_attention_on_dequantized_rows():
    n, hq, hkv, d, bs = 40, 8, 2, 128, 16
    full = wl.make_multi_case("f3", 3, [0], [n], hq, hkv, d, bs)
    ks, vs = np.array([0.02, 0.03]), np.array([0.025, 0.015])
    kq, vq = quantized(full, ks, vs)
    bt = full.block_tables.numpy()
    K = oracle.e4m3_decode(pa.gather_sequence(kq, bt[0], n)) * ks[:, None]
    V = oracle.e4m3_decode(pa.gather_sequence(vq, bt[0], n)) * vs[:, None]
    Q = pa.bf16_bits_to_f64(wl.bits(full.q))
    q = torch.from_numpy(Q).permute(1, 0, 2)[None]
    k = torch.from_numpy(K).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    v = torch.from_numpy(V).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    mask = torch.ones(n, n, dtype=torch.bool).tril()
    want = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=full.scale)[0].permute(1, 0, 2).numpy()
    a = 0
    for c in [16, 9, 15]:
        got = oracle.decode_multi_fp8(wl.bits(full.q)[a:a + c], kq, vq, ks, vs, bt,
                                      np.array([a + c]), np.array([0, c]), full.scale)
        assert np.abs(got - want[a:a + c]).max() < 1e-12, a
        a += c


def test_swapped_scales_are_rejected():
    case = wl.make_multi_case("f4", 4, [30, 7], [4, 4], 8, 2, 128, 16)
    ks, vs = np.array([0.03, 0.05]), np.array([0.01, 0.02])
    kq, vq = quantized(case, ks, vs)
    args = (case.block_tables.numpy(), case.context_lens.numpy(), case.q_start.numpy(),
            case.scale)
    right = oracle.decode_multi_fp8(wl.bits(case.q), kq, vq, ks, vs, *args)
    wrong = oracle.decode_multi_fp8(wl.bits(case.q), kq, vq, vs, ks, *args)
    assert np.abs(right - wrong).max() > 1e-3
