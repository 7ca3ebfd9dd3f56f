"""GPU parity for prefix sharing with copy-on-write.

* pa_copy_blocks against the oracle's block copy, bit for bit (bf16 and e4m3
  pools, many copies, ragged counts), and its skipping of ids outside the pool.
* A serving trace end to end: requests sharing a system prompt are admitted
  through the native prefix cache, their uncached positions are written by
  pa_kv_append after the device copies the cache asks for, sequences are
  forked and released, and fused decode steps (pa_prefix_append_tokens ->
  pa_copy_blocks -> pa_append_decode) run over the cache's tables. Each
  token's K/V row is a fixed function of (token id, position), so what every
  sequence must see is known without the pool: outputs are compared with the
  fp64 oracle over contiguous copies of those rows, and the pool read through
  every live table must hold exactly those rows.
"""

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from oracle import prefix_cache as pc
from paged_kv_cache_45_gb300 import binding as b
from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


def _copies(rng, nb, n):
    ids = rng.permutation(np.arange(1, nb))[:2 * n]
    return ids[:n].astype(np.int32), ids[n:2 * n].astype(np.int32)


@pytest.mark.parametrize("dtype,n", [(torch.bfloat16, 1), (torch.bfloat16, 37),
                                     (torch.bfloat16, 300), (torch.uint8, 45)])
def test_copy_blocks_bit_exact(cuda_lib, dtype, n):
    g = torch.Generator().manual_seed(n)
    nb, bs, hkv, d = 700, 16, 8, 128
    shape = (nb, bs, hkv, d)
    if dtype == torch.uint8:
        k = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
        v = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)
    else:
        k = torch.randn(shape, generator=g).to(dtype)
        v = torch.randn(shape, generator=g).to(dtype)
    src, dst = _copies(np.random.default_rng(n), nb, n)
    kd, vd = k.cuda(), v.cuda()
    b.pa_copy_blocks(kd, vd, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    torch.cuda.synchronize()
    kw = k.view(torch.uint8).numpy().copy() if dtype == torch.uint8 else wl.bits(k).copy()
    vw = v.view(torch.uint8).numpy().copy() if dtype == torch.uint8 else wl.bits(v).copy()
    pc.copy_blocks(kw, vw, list(zip(src.tolist(), dst.tolist())))
    got_k = kd.cpu().numpy() if dtype == torch.uint8 else wl.bits(kd.cpu())
    got_v = vd.cpu().numpy() if dtype == torch.uint8 else wl.bits(vd.cpu())
    assert np.array_equal(got_k, kw) and np.array_equal(got_v, vw)


def test_copy_blocks_skips_ids_outside_the_pool(cuda_lib):
    nb = 32
    k = torch.randn(nb, 4, 2, 64).to(torch.bfloat16)
    v = torch.randn(nb, 4, 2, 64).to(torch.bfloat16)
    kd, vd = k.cuda(), v.cuda()
    src = torch.tensor([3, -1, 40, 5], dtype=torch.int32)
    dst = torch.tensor([7, 8, 9, nb], dtype=torch.int32)
    b.pa_copy_blocks(kd, vd, src.cuda(), dst.cuda())
    torch.cuda.synchronize()
    kw, vw = wl.bits(k).copy(), wl.bits(v).copy()
    pc.copy_blocks(kw, vw, [(3, 7)])
    assert np.array_equal(wl.bits(kd.cpu()), kw) and np.array_equal(wl.bits(vd.cpu()), vw)


class RowTable:
    """K/V row of (token, position): bf16(T[token] + P[position]), fixed."""

    def __init__(self, vocab, max_pos, hkv, d, seed):
        g = torch.Generator().manual_seed(seed)
        self.tk = torch.randn(vocab, hkv, d, generator=g)
        self.tv = torch.randn(vocab, hkv, d, generator=g)
        self.pk = 0.5 * torch.randn(max_pos, hkv, d, generator=g)
        self.pv = 0.5 * torch.randn(max_pos, hkv, d, generator=g)

    def rows(self, tokens, positions):
        t = torch.as_tensor(tokens, dtype=torch.long)
        p = torch.as_tensor(positions, dtype=torch.long)
        return ((self.tk[t] + self.pk[p]).to(torch.bfloat16),
                (self.tv[t] + self.pv[p]).to(torch.bfloat16))


def _expected_out(rows, seq_tokens, q, scale, hkv, d):
    """fp64 oracle decode over contiguous private copies of each sequence's rows."""
    B = len(seq_tokens)
    bs = 16
    mb = max(-(-len(t) // bs) for t in seq_tokens)
    kc = np.zeros((B * mb + 1, bs, hkv, d), dtype=np.uint16)
    vc = np.zeros_like(kc)
    tables = np.zeros((B, mb), dtype=np.int32)
    for i, toks in enumerate(seq_tokens):
        k, v = rows.rows(toks, range(len(toks)))
        n = len(toks)
        flat_k = np.zeros((mb * bs, hkv, d), dtype=np.uint16)
        flat_v = np.zeros_like(flat_k)
        flat_k[:n], flat_v[:n] = wl.bits(k), wl.bits(v)
        kc[1 + i * mb:1 + (i + 1) * mb] = flat_k.reshape(mb, bs, hkv, d)
        vc[1 + i * mb:1 + (i + 1) * mb] = flat_v.reshape(mb, bs, hkv, d)
        tables[i] = 1 + i * mb + np.arange(mb)
    lens = np.array([len(t) for t in seq_tokens], dtype=np.int32)
    return pa.decode(wl.bits(q), kc, vc, tables, lens, scale)


def test_serving_trace_with_shared_prefixes_and_forks(cuda_lib):
    hq, hkv, d, bs, nb = 16, 2, 128, 16, 600
    vocab, scale = 64, 1.0 / np.sqrt(128)
    rng = np.random.default_rng(7)
    rows = RowTable(vocab, 4096, hkv, d, seed=3)
    kd = wl.nan_pool(nb, bs, hkv, d).cuda()
    vd = wl.nan_pool(nb, bs, hkv, d).cuda()
    cache = b.PrefixCache(nb, bs)
    system = list(rng.integers(0, vocab, 3 * bs + 5))
    live = {}                                    # seq id -> tokens
    n_copies = 0
    n_hits = 0

    def device_copies(src, dst):
        nonlocal n_copies
        if len(src):
            n_copies += len(src)
            b.pa_copy_blocks(kd, vd, torch.as_tensor(np.asarray(src, np.int32)).cuda(),
                             torch.as_tensor(np.asarray(dst, np.int32)).cuda())

    def admit(tokens):
        nonlocal n_hits
        sid, cached = cache.admit(tokens)
        n_hits += cached > 0
        slots, copies = cache.write_slots(sid, cached, len(tokens))
        device_copies([c[0] for c in copies], [c[1] for c in copies])
        k, v = rows.rows(tokens[cached:], range(cached, len(tokens)))
        b.pa_kv_append(k.cuda(), v.cuda(), torch.as_tensor(slots, dtype=torch.int64).cuda(),
                       kd, vd)
        live[sid] = list(tokens)
        return sid

    first = admit(system + list(rng.integers(0, vocab, 9)))
    cache.release(first, live.pop(first))        # the system prompt is now cached
    for k in range(10):
        admit(system + list(rng.integers(0, vocab, int(rng.integers(0, 40)))))
    admit(system[:3 * bs])                       # whole prompt cached: one token given back
    for step in range(8):
        if step in (2, 5):                       # forks share their parent's partial block
            parent = list(live)[int(rng.integers(0, len(live)))]
            live[cache.fork(parent)] = list(live[parent])
        if step in (3, 6):                       # a finished request feeds the cache
            sid = list(live)[0]
            cache.release(sid, live.pop(sid))
            admit(system + list(rng.integers(0, vocab, 20)))
        sids = list(live)
        new_tok = [int(x) for x in rng.integers(0, vocab, len(sids))]
        slots, (src, dst) = cache.append_tokens(sids)
        device_copies(src, dst)
        for sid, t in zip(sids, new_tok):
            live[sid].append(t)
        pos = [len(live[s]) - 1 for s in sids]
        k_new, v_new = rows.rows(new_tok, pos)
        mb = max(len(cache.table(s)) for s in sids)
        tables, lens = cache.tables(sids, mb)
        q = torch.randn(len(sids), hq, d, generator=torch.Generator().manual_seed(step)).to(
            torch.bfloat16)
        ws = torch.zeros(b.pa_decode_balanced_workspace_bytes(len(sids), hkv, d),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty(len(sids), hq, d, dtype=torch.bfloat16, device="cuda")
        b.pa_append_decode(q.cuda(), k_new.cuda(), v_new.cuda(),
                           torch.as_tensor(slots, dtype=torch.int64).cuda(), kd, vd,
                           torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                           scale, ws, out)
        want = _expected_out(rows, [live[s] for s in sids], q, scale, hkv, d)
        P.assert_close(P.to_f64(out), want, f"step {step}")
    assert n_hits >= 10 and n_copies >= 3
    torch.cuda.synchronize()
    kh, vh = wl.bits(kd.cpu()), wl.bits(vd.cpu())
    for sid, toks in live.items():               # the pool holds every sequence's rows
        t = cache.table(sid)
        k, v = rows.rows(toks, range(len(toks)))
        n = len(toks)
        got_k = kh[t].reshape(-1, hkv, d)[:n]
        got_v = vh[t].reshape(-1, hkv, d)[:n]
        assert np.array_equal(got_k, wl.bits(k)) and np.array_equal(got_v, wl.bits(v)), sid
    assert b.pa_last_device_error() == 0
