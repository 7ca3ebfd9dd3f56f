"""Guard canaries: no entry point writes outside the buffers it is given.

Every device buffer an entry point writes (outputs, fixed-split partials and
row lengths, the balanced workspaces, the K/V pools) is carved out of a
larger allocation with GUARD bytes before and after it, filled with a fixed
byte pattern. Each entry point then runs on small ragged cases (block sizes
1 / 8 / 16 / 32, GQA groups 1 / 2 / 8, head_dim 64 and 128, with and without
context splits) and the guards must still hold the pattern bit for bit. The
main outputs are also checked against the fp64 oracle at the parity bar of
the other tests, so a kernel that wrote nothing could not pass.
"""

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side (keeps the buffer 256-byte aligned)
PATTERN = 0xA5
LENS = [0, 1, 2, 17, 33, 100, 257, 600]


class Guarded:
    """A device tensor of `shape`/`dtype` between two guard regions."""

    def __init__(self, shape, dtype, init=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)
        if init is not None:
            self.t.copy_(init.to(device="cuda", dtype=dtype) if torch.is_tensor(init)
                         else torch.full(shape, init, dtype=dtype))

    def check(self, what):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        assert bool((head == PATTERN).all()), f"{what}: bytes before the buffer were written"
        assert bool((tail == PATTERN).all()), f"{what}: bytes after the buffer were written"


def _pool(t):
    return Guarded(tuple(t.shape), t.dtype, t)


def _ws(nbytes):
    return Guarded((nbytes,), torch.uint8, 0)


SHAPES = [(bs, d, hq, hkv) for bs in (1, 8, 16, 32) for d in (64, 128)
          for hq, hkv in ((2, 2), (4, 2), (16, 2))]


def _id(s):
    return f"bs{s[0]}-d{s[1]}-g{s[2] // s[3]}"


@pytest.mark.parametrize("shape", SHAPES, ids=[_id(s) for s in SHAPES])
def test_decode_entry_points_stay_inside_their_buffers(cuda_lib, shape):
    b = cuda_lib
    bs, d, hq, hkv = shape
    case = wl.make_case("guard", 900 + bs + d + hq, LENS, hq, hkv, d, bs)
    B = case.batch
    q = case.q.cuda()
    tables, lens = case.block_tables.cuda(), case.context_lens.cuda()
    kn, vn, slots = case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda()
    ref = P.oracle_out(case)

    # append, then every decode form over the appended pool
    kc, vc = _pool(case.k_cache), _pool(case.v_cache)
    b.pa_kv_append(kn, vn, slots, kc.t, vc.t)
    out = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode(q, kc.t, vc.t, tables, lens, case.scale, out.t)
    split = 64
    S = b.pa_decode_num_splits(case.max_blocks * bs, split)
    po = Guarded((B, hq, S, d), torch.float32, float("nan"))
    pl = Guarded((B, hq, S), torch.float32, float("nan"))
    out_s = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode(q, kc.t, vc.t, tables, lens, case.scale, out_s.t, split, S, po.t, pl.t)
    b.pa_decode_splitk_reduce(po.t, pl.t, lens, split, out_s.t)
    ws_bytes = b.pa_decode_balanced_workspace_bytes(B, hkv, d)
    ws = _ws(ws_bytes)
    out_b = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode_balanced(q, kc.t, vc.t, tables, lens, case.scale, ws.t, out_b.t)
    out_st = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode_balanced_static(q, kc.t, vc.t, tables, lens, case.scale, out_st.t)

    # the fused step on fresh pools
    kf, vf = _pool(case.k_cache), _pool(case.v_cache)
    ws_f = _ws(ws_bytes)
    out_f = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_append_decode(q, kn, vn, slots, kf.t, vf.t, tables, lens, case.scale, ws_f.t, out_f.t)
    torch.cuda.synchronize()

    for g, what in ((kc, "k_cache (append)"), (vc, "v_cache (append)"), (out, "pa_decode out"),
                    (po, "part_out"), (pl, "part_lse"), (out_s, "reduce out"),
                    (ws, "balanced workspace"), (out_b, "balanced out"),
                    (out_st, "static-scratch out"), (kf, "k_cache (fused)"),
                    (vf, "v_cache (fused)"), (ws_f, "fused workspace"), (out_f, "fused out")):
        g.check(what)
    for g, what in ((out, "pa_decode"), (out_s, "split + reduce"), (out_b, "balanced"),
                    (out_st, "static scratch"), (out_f, "fused step")):
        P.assert_close(P.to_f64(g.t), ref, what)
    assert b.pa_last_device_error() == 0


FP8_SHAPES = [(bs, hq, hkv) for bs in (1, 8, 16, 32) for hq, hkv in ((2, 2), (4, 2), (16, 2))]


@pytest.mark.parametrize("shape", FP8_SHAPES, ids=[f"bs{s[0]}-g{s[1] // s[2]}" for s in FP8_SHAPES])
def test_fp8_entry_points_stay_inside_their_buffers(cuda_lib, shape):
    b = cuda_lib
    bs, hq, hkv = shape
    d = 128
    case = wl.make_case("guard8", 950 + bs + hq, LENS, hq, hkv, d, bs)
    f8 = wl.fp8_pool(case, 5)
    B = case.batch
    q = case.q.cuda()
    tables, lens = case.block_tables.cuda(), case.context_lens.cuda()
    kn, vn, slots = case.k_new.cuda(), case.v_new.cuda(), case.slot_mapping.cuda()
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    kcodes, vcodes = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    pa.kv_append_fp8_inplace(kcodes, vcodes, wl.bits(case.k_new), wl.bits(case.v_new),
                             case.slot_mapping.numpy(), f8["k_scale"].numpy(),
                             f8["v_scale"].numpy())
    ref = pa.decode_fp8(wl.bits(case.q), kcodes, vcodes, f8["k_scale"].numpy(),
                        f8["v_scale"].numpy(), case.block_tables.numpy(),
                        case.context_lens.numpy(), case.scale)

    kc, vc = _pool(f8["k_codes"]), _pool(f8["v_codes"])
    b.pa_kv_append_fp8(kn, vn, slots, kc.t, vc.t, ks, vs)
    ws_bytes = b.pa_decode_balanced_workspace_bytes(B, hkv, d)
    ws = _ws(ws_bytes)
    out = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode_balanced_fp8(q, kc.t, vc.t, ks, vs, tables, lens, case.scale, ws.t, out.t)
    kf, vf = _pool(f8["k_codes"]), _pool(f8["v_codes"])
    ws_f = _ws(ws_bytes)
    out_f = Guarded((B, hq, d), torch.bfloat16, float("nan"))
    b.pa_append_decode_fp8(q, kn, vn, slots, kf.t, vf.t, ks, vs, tables, lens, case.scale,
                           ws_f.t, out_f.t)
    torch.cuda.synchronize()
    for g, what in ((kc, "k codes (append)"), (vc, "v codes (append)"), (ws, "workspace"),
                    (out, "out"), (kf, "k codes (fused)"), (vf, "v codes (fused)"),
                    (ws_f, "fused workspace"), (out_f, "fused out")):
        g.check(what)
    assert np.array_equal(kc.t.cpu().numpy(), kcodes)
    assert np.array_equal(vf.t.cpu().numpy(), vcodes)
    P.assert_close(P.to_f64(out.t), ref, "fp8 balanced")
    P.assert_close(P.to_f64(out_f.t), ref, "fp8 fused step")
    assert b.pa_last_device_error() == 0


MULTI_SHAPES = [(bs, d, hq, hkv, qlen) for bs in (1, 8, 16, 32) for d in (64, 128)
                for hq, hkv, qlen in ((4, 2, 5), (16, 2, 3), (16, 2, 40))]


@pytest.mark.parametrize("shape", MULTI_SHAPES,
                         ids=[f"bs{s[0]}-d{s[1]}-g{s[2] // s[3]}-n{s[4]}" for s in MULTI_SHAPES])
def test_multi_token_entry_points_stay_inside_their_buffers(cuda_lib, shape):
    b = cuda_lib
    bs, d, hq, hkv, qlen = shape
    ctx0 = [0, 3, 30, 129, 400]
    qlens = [qlen, 1, qlen, max(1, qlen - 2), qlen]
    mc = wl.make_multi_case("guardm", 970 + bs + d + qlen, ctx0, qlens, hq, hkv, d, bs)
    R, B = int(mc.q.shape[0]), mc.batch
    kc, vc = _pool(mc.k_cache), _pool(mc.v_cache)
    b.pa_kv_append(mc.k_new.cuda(), mc.v_new.cuda(), mc.slot_mapping.cuda(), kc.t, vc.t)
    q, tables, lens = mc.q.cuda(), mc.block_tables.cuda(), mc.context_lens.cuda()
    qs = mc.q_start.cuda()
    out = Guarded((R, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode_multi(q, kc.t, vc.t, tables, lens, qs, mc.max_q_len, mc.scale, out.t)
    guards = [(kc, "k_cache"), (vc, "v_cache"), (out, "multi out")]
    outs = [(out, "multi")]
    if mc.max_q_len * (hq // hkv) <= 64:  # short chunks: split and balanced forms
        # split 64 runs the column-warp kernel; split 128 the tcgen05 one where
        # it applies (head_dim 128, block size >= 8, <= 32 columns a KV head)
        for split in (64, 128):
            S = b.pa_decode_num_splits(int(mc.block_tables.shape[1]) * bs, split)
            po = Guarded((R, hq, S, d), torch.float32, float("nan"))
            pl = Guarded((R, hq, S), torch.float32, float("nan"))
            rl = Guarded((R,), torch.int32, -7)
            out_s = Guarded((R, hq, d), torch.bfloat16, float("nan"))
            b.pa_decode_multi(q, kc.t, vc.t, tables, lens, qs, mc.max_q_len, mc.scale, out_s.t,
                              split, S, po.t, pl.t, rl.t)
            b.pa_decode_splitk_reduce(po.t, pl.t, rl.t, split, out_s.t)
            guards += [(po, f"part_out, split {split}"), (pl, f"part_lse, split {split}"),
                       (rl, f"row_lens, split {split}"), (out_s, f"reduce out, split {split}")]
            outs += [(out_s, f"multi split {split} + reduce")]
        ws = _ws(b.pa_decode_multi_balanced_workspace_bytes(B, hkv, d))
        out_b = Guarded((R, hq, d), torch.bfloat16, float("nan"))
        b.pa_decode_multi_balanced(q, kc.t, vc.t, tables, lens, qs, mc.max_q_len, mc.scale,
                                   ws.t, out_b.t)
        guards += [(ws, "multi workspace"), (out_b, "multi balanced out")]
        outs += [(out_b, "multi balanced")]
    torch.cuda.synchronize()
    for g, what in guards:
        g.check(what)
    kmo, vmo = pa.kv_append(wl.bits(mc.k_cache), wl.bits(mc.v_cache), wl.bits(mc.k_new),
                            wl.bits(mc.v_new), mc.slot_mapping.numpy())
    ref = pa.decode_multi(wl.bits(mc.q), kmo, vmo, mc.block_tables.numpy(),
                          mc.context_lens.numpy(), mc.q_start.numpy(), mc.scale)
    for g, what in outs:
        P.assert_close(P.to_f64(g.t), ref, what)
    assert b.pa_last_device_error() == 0


@pytest.mark.parametrize("bs", [1, 8, 16, 32])
def test_fp8_multi_token_stays_inside_its_buffers(cuda_lib, bs):
    b = cuda_lib
    hq, hkv, d = 16, 2, 128
    mc = wl.make_multi_case("guardm8", 990 + bs, [0, 3, 30, 129, 400], [4, 1, 4, 2, 4], hq, hkv,
                            d, bs)
    f8 = wl.fp8_pool(mc, 6)
    R = int(mc.q.shape[0])
    kc, vc = _pool(f8["k_codes"]), _pool(f8["v_codes"])
    ks, vs = f8["k_scale"].cuda(), f8["v_scale"].cuda()
    b.pa_kv_append_fp8(mc.k_new.cuda(), mc.v_new.cuda(), mc.slot_mapping.cuda(), kc.t, vc.t,
                       ks, vs)
    q, tables, lens, qs = (mc.q.cuda(), mc.block_tables.cuda(), mc.context_lens.cuda(),
                           mc.q_start.cuda())
    out = Guarded((R, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode_multi_fp8(q, kc.t, vc.t, ks, vs, tables, lens, qs, mc.max_q_len, mc.scale,
                          out.t)
    split = 64
    S = b.pa_decode_num_splits(int(mc.block_tables.shape[1]) * bs, split)
    po = Guarded((R, hq, S, d), torch.float32, float("nan"))
    pl = Guarded((R, hq, S), torch.float32, float("nan"))
    rl = Guarded((R,), torch.int32, -7)
    out_s = Guarded((R, hq, d), torch.bfloat16, float("nan"))
    b.pa_decode_multi_fp8(q, kc.t, vc.t, ks, vs, tables, lens, qs, mc.max_q_len, mc.scale,
                          out_s.t, split, S, po.t, pl.t, rl.t)
    b.pa_decode_splitk_reduce(po.t, pl.t, rl.t, split, out_s.t)
    torch.cuda.synchronize()
    for g, what in ((kc, "k codes"), (vc, "v codes"), (out, "out"), (po, "part_out"),
                    (pl, "part_lse"), (rl, "row_lens"), (out_s, "reduce out")):
        g.check(what)
    kcodes, vcodes = f8["k_codes"].numpy().copy(), f8["v_codes"].numpy().copy()
    pa.kv_append_fp8_inplace(kcodes, vcodes, wl.bits(mc.k_new), wl.bits(mc.v_new),
                             mc.slot_mapping.numpy(), f8["k_scale"].numpy(),
                             f8["v_scale"].numpy())
    ref = pa.decode_multi_fp8(wl.bits(mc.q), kcodes, vcodes, f8["k_scale"].numpy(),
                              f8["v_scale"].numpy(), mc.block_tables.numpy(),
                              mc.context_lens.numpy(), mc.q_start.numpy(), mc.scale)
    P.assert_close(P.to_f64(out.t), ref, "fp8 multi")
    P.assert_close(P.to_f64(out_s.t), ref, "fp8 multi split + reduce")
    assert b.pa_last_device_error() == 0


def test_copy_blocks_stays_inside_the_pool(cuda_lib):
    b = cuda_lib
    nb, bs, hkv, d = 64, 16, 2, 128
    g = torch.Generator().manual_seed(3)
    k = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nb, bs, hkv, d, generator=g).to(torch.bfloat16)
    kc, vc = _pool(k), _pool(v)
    # the first and last blocks as destinations, ids past the pool skipped
    src = torch.tensor([5, 7, 9, 70], dtype=torch.int32, device="cuda")
    dst = torch.tensor([0, nb - 1, 12, 3], dtype=torch.int32, device="cuda")
    b.pa_copy_blocks(kc.t, vc.t, src, dst)
    torch.cuda.synchronize()
    kc.check("k_cache")
    vc.check("v_cache")
    want = k.clone()
    want[0], want[nb - 1], want[12] = k[5], k[7], k[9]
    assert torch.equal(kc.t.cpu().view(torch.int16), want.view(torch.int16))
