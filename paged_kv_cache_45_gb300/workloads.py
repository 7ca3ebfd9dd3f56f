"""Seeded synthetic inputs for paged-KV decode attention.

These generators serve both the CPU oracle (through the tests) and the CUDA
path. They hold none of the attention arithmetic: they draw lengths, block
placements and N(0,1) values, and lay the drawn K/V rows into a paged pool
through the block tables a :class:`BlockAllocator` hands out.

Shapes follow the pages' model classes: the 8B class (32 query heads, 8 KV
heads, head_dim 128) and the 70B class (64 query heads, 8 KV heads, head_dim
128), bf16, block_size 16 ("Text Generation Inference: Hugging Face's
production-grade LLM inference server", section "Production Pattern: KV Cache
Math"; "The inference request lifecycle", section "Work the GQA number before
choosing concurrency").

Recipe (every draw is seeded):

* lengths and block ids: ``numpy.random.Generator(PCG64(seed))``;
  "log-uniform [a, b]" is ``round(exp(U(ln a, ln b)))``;
* tensors: ``torch.randn`` on a CPU ``torch.Generator`` seeded from
  ``(seed, purpose)``, drawn in float32 and rounded to bfloat16 (RNE);
* every pool slot that holds no token of a live sequence, block 0 included,
  holds bfloat16 NaN, so a kernel that reads a slot it should not turns its
  output into NaN;
* ``context_lens`` are counted after the step's append: the appended token is
  attended over by the same step.
"""

from __future__ import annotations

import math
import time
from dataclasses import dataclass, field

import numpy as np
import torch

from .allocator import BlockAllocator

BF16_NAN_BITS = 0x7FC0


# ---------------------------------------------------------------------------
# small helpers
# ---------------------------------------------------------------------------

def bits(t: torch.Tensor) -> np.ndarray:
    """``uint16`` NumPy view of a bfloat16 CPU tensor (no copy when contiguous)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bfloat16 tensor")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _torch_gen(seed: int, purpose: int) -> torch.Generator:
    return torch.Generator().manual_seed((int(seed) * 1_000_003 + int(purpose)) % (2 ** 63))


def randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def loguniform(rng: np.random.Generator, lo: float, hi: float, n: int) -> np.ndarray:
    return np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), n))).astype(np.int64)


def nan_pool(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int) -> torch.Tensor:
    t = torch.full((num_blocks, block_size, num_kv_heads, head_dim), BF16_NAN_BITS,
                   dtype=torch.int16)
    return t.view(torch.bfloat16)


def poison_blocks(cache: torch.Tensor, blocks) -> None:
    """Fill whole physical blocks with bfloat16 NaN (CPU or device tensor)."""
    if len(blocks) == 0:
        return
    idx = torch.as_tensor(list(blocks), dtype=torch.long, device=cache.device)
    cache.view(torch.int16)[idx] = BF16_NAN_BITS


def token_rows(blocks, n_tokens: int, block_size: int, start: int = 0) -> np.ndarray:
    """Flat pool rows (``block * block_size + offset``) of logical tokens
    ``start .. start + n_tokens - 1`` of a sequence owning ``blocks``."""
    t = np.arange(start, start + n_tokens, dtype=np.int64)
    blk = np.asarray(blocks, dtype=np.int64)
    return blk[t // block_size] * block_size + t % block_size


def pad_tables(seq_blocks, max_blocks: int) -> torch.Tensor:
    tab = np.zeros((len(seq_blocks), max_blocks), dtype=np.int32)
    for b, blks in enumerate(seq_blocks):
        if len(blks) > max_blocks:
            raise ValueError("sequence owns more blocks than the table holds")
        tab[b, :len(blks)] = blks
    return torch.from_numpy(tab)


# ---------------------------------------------------------------------------
# one decode step over a paged pool
# ---------------------------------------------------------------------------

@dataclass
class DecodeCase:
    """Inputs of one append + decode step. Caches hold the state *before* the
    append; ``context_lens`` count the tokens attended over *after* it."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    q: torch.Tensor                 # bf16 [B, Hq, D]
    k_cache: torch.Tensor           # bf16 [NB, bs, Hkv, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # int32 [B, MB]
    context_lens: torch.Tensor      # int32 [B]
    k_new: torch.Tensor | None = None       # bf16 [T, Hkv, D]
    v_new: torch.Tensor | None = None
    slot_mapping: torch.Tensor | None = None  # int64 [T]
    split_tokens: int = 0           # suggested context split (0: none)
    seq_blocks: list = field(default_factory=list)
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])


def make_case(name: str, seed: int, ctx_before, num_q_heads: int, num_kv_heads: int,
              head_dim: int, block_size: int, *, append: bool = True,
              num_blocks: int | None = None, spare_frac: float = 0.10,
              max_blocks: int | None = None, shared_prefix: int = 0,
              k_outlier_frac: float = 0.0, k_outlier_mul: float = 8.0,
              split_tokens: int = 0, scale: float | None = None) -> DecodeCase:
    """Build a seeded decode step.

    ``ctx_before[b]`` tokens of sequence ``b`` are cached already; with
    ``append`` one new token per sequence is written by the step and attended
    over (``context_lens = ctx_before + 1``). Physical blocks leave a shuffled
    free list (block 0 reserved). ``shared_prefix`` tokens (a multiple of
    ``block_size``) are held in the same physical blocks by every sequence,
    refcounted. ``k_outlier_frac`` of each sequence's positions have their
    whole K row multiplied by ``k_outlier_mul`` before the bf16 rounding.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx0 = np.asarray(ctx_before, dtype=np.int64)
    B = len(ctx0)
    ctx1 = ctx0 + (1 if append else 0)
    bs = block_size
    if shared_prefix % bs:
        raise ValueError("shared prefix must fill whole blocks")
    if np.any(ctx0 < shared_prefix):
        raise ValueError("every sequence must contain the shared prefix")
    n_pref = shared_prefix // bs
    need = [-(-int(c) // bs) for c in ctx1]
    private = sum(n - n_pref for n in need) + n_pref
    if num_blocks is None:
        num_blocks = int(math.ceil((1.0 + spare_frac) * private)) + 1
    if num_blocks - 1 < private:
        raise ValueError("pool too small for the requested lengths")
    order = 1 + rng.permutation(num_blocks - 1)
    alloc = BlockAllocator(num_blocks, order=order)
    prefix_blocks = alloc.allocate(n_pref) if n_pref else []
    if n_pref and B > 1:
        for _ in range(B - 1):
            alloc.share(prefix_blocks)
    seq_blocks = [prefix_blocks + alloc.allocate(n - n_pref) for n in need]
    if max_blocks is None:
        max_blocks = max(max(need), 1)

    H, D = num_kv_heads, head_dim
    k_cache = nan_pool(num_blocks, bs, H, D)
    v_cache = nan_pool(num_blocks, bs, H, D)
    kflat, vflat = k_cache.view(-1, H, D), v_cache.view(-1, H, D)

    gk, gv, gq, gn = (_torch_gen(seed, p) for p in (1, 2, 3, 4))
    # shared prefix rows, drawn once
    if shared_prefix:
        rows = token_rows(prefix_blocks, shared_prefix, bs)
        kflat[rows] = randn_bf16(gk, (shared_prefix, H, D))
        vflat[rows] = randn_bf16(gv, (shared_prefix, H, D))
    for b in range(B):
        n_priv = int(ctx0[b]) - shared_prefix
        if n_priv <= 0:
            continue
        rows = token_rows(seq_blocks[b], n_priv, bs, start=shared_prefix)
        kv = torch.randn((n_priv, H, D), generator=gk, dtype=torch.float32)
        if k_outlier_frac > 0:
            n_out = int(math.floor(k_outlier_frac * int(ctx0[b])))
            pos = rng.choice(n_priv, size=n_out, replace=False)
            kv[torch.from_numpy(pos)] *= k_outlier_mul
        kflat[rows] = kv.to(torch.bfloat16)
        vflat[rows] = randn_bf16(gv, (n_priv, H, D))

    q = randn_bf16(gq, (B, num_q_heads, D))
    k_new = v_new = slots = None
    if append:
        k_new = randn_bf16(gn, (B, H, D))
        v_new = randn_bf16(gn, (B, H, D))
        slots = torch.from_numpy(np.array(
            [int(token_rows(seq_blocks[b], 1, bs, start=int(ctx0[b]))[0]) for b in range(B)],
            dtype=np.int64))
    return DecodeCase(
        name=name, num_q_heads=num_q_heads, num_kv_heads=H, head_dim=D, block_size=bs,
        num_blocks=num_blocks, scale=(1.0 / math.sqrt(D)) if scale is None else scale,
        q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=pad_tables(seq_blocks, max_blocks),
        context_lens=torch.from_numpy(ctx1.astype(np.int32)),
        k_new=k_new, v_new=v_new, slot_mapping=slots, split_tokens=split_tokens,
        seq_blocks=seq_blocks,
        meta={"seed": seed, "ctx_before": ctx0.tolist(), "shared_prefix": shared_prefix})


# ---------------------------------------------------------------------------
# several new query tokens per sequence (chunked prefill, speculative verify)
# ---------------------------------------------------------------------------

@dataclass
class MultiCase:
    """Inputs of one step in which sequence ``b`` appends ``q_len[b]`` tokens
    and queries with all of them. Query and new K/V rows are packed: sequence
    ``b`` owns rows ``q_start[b] .. q_start[b+1]-1``. Caches hold the state
    before the append; ``context_lens`` count tokens after it."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    q: torch.Tensor                 # bf16 [R, Hq, D]
    q_start: torch.Tensor           # int32 [B + 1]
    k_cache: torch.Tensor           # bf16 [NB, bs, Hkv, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # int32 [B, MB]
    context_lens: torch.Tensor      # int32 [B]
    k_new: torch.Tensor             # bf16 [R, Hkv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # int64 [R]
    seq_blocks: list = field(default_factory=list)

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_q_len(self) -> int:
        qs = self.q_start.numpy()
        return int((qs[1:] - qs[:-1]).max()) if self.batch else 0


def make_multi_case(name: str, seed: int, ctx_before, q_lens, num_q_heads: int,
                    num_kv_heads: int, head_dim: int, block_size: int, *,
                    spare_frac: float = 0.10, scale: float | None = None) -> MultiCase:
    """Seeded step with ``q_lens[b]`` new tokens after ``ctx_before[b]`` cached
    ones. Blocks come off a shuffled free list (block 0 reserved); every slot
    nobody owns is NaN."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx0 = np.asarray(ctx_before, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    B = len(ctx0)
    ctx1 = ctx0 + ql
    bs = block_size
    need = [-(-int(c) // bs) for c in ctx1]
    num_blocks = int(math.ceil((1.0 + spare_frac) * sum(need))) + 1
    order = 1 + rng.permutation(num_blocks - 1)
    alloc = BlockAllocator(num_blocks, order=order)
    seq_blocks = [alloc.allocate(n) for n in need]
    H, D = num_kv_heads, head_dim
    k_cache = nan_pool(num_blocks, bs, H, D)
    v_cache = nan_pool(num_blocks, bs, H, D)
    kflat, vflat = k_cache.view(-1, H, D), v_cache.view(-1, H, D)
    gk, gv, gq, gn = (_torch_gen(seed, p) for p in (11, 12, 13, 14))
    for b in range(B):
        n = int(ctx0[b])
        if n:
            rows = token_rows(seq_blocks[b], n, bs)
            kflat[rows] = randn_bf16(gk, (n, H, D))
            vflat[rows] = randn_bf16(gv, (n, H, D))
    R = int(ql.sum())
    q_start = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    slots = np.concatenate([token_rows(seq_blocks[b], int(ql[b]), bs, start=int(ctx0[b]))
                            for b in range(B)] + [np.zeros(0, dtype=np.int64)]).astype(np.int64)
    return MultiCase(
        name=name, num_q_heads=num_q_heads, num_kv_heads=H, head_dim=D, block_size=bs,
        num_blocks=num_blocks, scale=(1.0 / math.sqrt(D)) if scale is None else scale,
        q=randn_bf16(gq, (R, num_q_heads, D)), q_start=torch.from_numpy(q_start),
        k_cache=k_cache, v_cache=v_cache,
        block_tables=pad_tables(seq_blocks, max(max(need, default=1), 1)),
        context_lens=torch.from_numpy(ctx1.astype(np.int32)),
        k_new=randn_bf16(gn, (R, H, D)), v_new=randn_bf16(gn, (R, H, D)),
        slot_mapping=torch.from_numpy(slots), seq_blocks=seq_blocks)


def spec_verify_case(seed: int = 0, batch: int = 256, q_len: int = 4) -> MultiCase:
    """Speculative verification on the 70B shape: ``batch`` sequences with
    lengths log-uniform in [128, 8192], each checking ``q_len`` new tokens (the
    drafted ones plus one); 64 query heads on 8 KV heads, head_dim 128,
    block_size 16."""
    rng = np.random.Generator(np.random.PCG64(seed + 21_000))
    ctx = loguniform(rng, 128, 8192, batch)
    return make_multi_case(f"spec_b{batch}_q{q_len}", seed, ctx, [q_len] * batch, 64, 8, 128, 16)


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def tiny_case(seed: int = 0) -> DecodeCase:
    """4 sequences holding {1, 7, 16, 33} tokens before one appended token each;
    2 query heads on 1 KV head, head_dim 64, block_size 16, a 16-block pool
    placed by a seeded permutation, scale 1/sqrt(64)."""
    return make_case("tiny", seed, [1, 7, 16, 33], 2, 1, 64, 16, num_blocks=16,
                     scale=1.0 / 8.0)


def llama8b_case(seed: int = 0, batch: int = 64, ctx_lo: int = 512,
                 ctx_hi: int = 4096) -> DecodeCase:
    """8B-shape layer: 32 q heads, 8 KV heads, head_dim 128; ``batch`` sequences
    with lengths uniform in [ctx_lo, ctx_hi] before the append; the pool is the
    blocks needed plus 10% free, shuffled."""
    rng = np.random.Generator(np.random.PCG64(seed + 7_000))
    ctx = rng.integers(ctx_lo, ctx_hi, size=batch, endpoint=True)
    return make_case(f"8b_b{batch}", seed, ctx, 32, 8, 128, 16, spare_frac=0.10)


def long_context_case(seed: int = 0, batch: int = 4, ctx: int = 131072,
                      split_tokens: int = 4096, num_q_heads: int = 32) -> DecodeCase:
    """Long contexts, decode only (no append): ``batch`` sequences of exactly
    ``ctx`` tokens, 8B heads, 1% of each sequence's positions with K x8, split
    into ``split_tokens``-token ranges merged by log-sum-exp."""
    return make_case(f"long_{ctx}", seed, [ctx] * batch, num_q_heads, 8, 128, 16,
                     append=False, spare_frac=0.0, k_outlier_frac=0.01,
                     split_tokens=split_tokens)


def prefix_sharing_case(seed: int = 0, batch: int = 128, prefix: int = 2048,
                        suf_lo: int = 64, suf_hi: int = 1024) -> DecodeCase:
    """``batch`` sequences whose first ``prefix`` tokens are the same physical
    blocks in every block table (refcount ``batch``), then private suffixes of
    length uniform in [suf_lo, suf_hi] in shuffled private blocks; 8B heads."""
    rng = np.random.Generator(np.random.PCG64(seed + 9_000))
    suf = rng.integers(suf_lo, suf_hi, size=batch, endpoint=True)
    return make_case(f"prefix_b{batch}", seed, prefix + suf, 32, 8, 128, 16,
                     spare_frac=0.10, shared_prefix=prefix)


# ---------------------------------------------------------------------------
# 70B-shape continuous batching
# ---------------------------------------------------------------------------

@dataclass
class CBStep:
    """One continuous-batching iteration.

    ``freed``: blocks released by finished sequences (to be NaN-poisoned).
    ``fill_*``: prompt rows of joining sequences, written with the append
    kernel before the step (prefill stand-in, timed apart from the step).
    The rest is the decode step: one appended token per sequence, then
    attention over ``context_lens`` (after the append)."""
    index: int
    finished: list
    freed: list
    fill_slots: torch.Tensor        # int64 [P]
    fill_k: torch.Tensor            # bf16 [P, Hkv, D]
    fill_v: torch.Tensor
    slot_mapping: torch.Tensor      # int64 [B]
    k_new: torch.Tensor             # bf16 [B, Hkv, D]
    v_new: torch.Tensor
    q: torch.Tensor                 # bf16 [B, Hq, D]
    block_tables: torch.Tensor      # int32 [B, MB]
    context_lens: torch.Tensor      # int32 [B]


class ContinuousBatching:
    """70B-shape continuous batching: 64 q heads, 8 KV heads, head_dim 128,
    block_size 16, ``batch`` running sequences with lengths log-uniform in
    [ctx_lo, ctx_hi]. Each iteration every sequence finishes with probability
    ``p_finish`` (its blocks go back to the free list) and a newcomer with a
    prompt log-uniform in [prompt_lo, prompt_hi] takes its slot, its blocks
    from the free list; then one token is appended per sequence and decoded.

    The schedule (lengths, finishes, block ids) is drawn up front for
    ``iterations`` steps; tensors are drawn per iteration from generators
    seeded by (seed, iteration), so any iteration is reproducible alone.
    """

    def __init__(self, seed: int = 0, batch: int = 256, num_q_heads: int = 64,
                 num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                 iterations: int = 32, p_finish: float = 0.02,
                 ctx_lo: int = 128, ctx_hi: int = 8192,
                 prompt_lo: int = 128, prompt_hi: int = 2048):
        self.seed = seed
        self.B, self.Hq, self.Hkv, self.D, self.bs = batch, num_q_heads, num_kv_heads, head_dim, block_size
        self.iterations = iterations
        self.scale = 1.0 / math.sqrt(head_dim)
        rng = np.random.Generator(np.random.PCG64(seed + 3_000))
        bs = block_size
        ctx0 = loguniform(rng, ctx_lo, ctx_hi, batch)
        initial_blocks = int(sum(-(-int(c) // bs) for c in ctx0))
        self.num_blocks = int(math.ceil(1.25 * initial_blocks)) + 3 * batch
        self.max_blocks = -(-(max(ctx_hi, prompt_hi) + iterations + 1) // bs)
        order = 1 + rng.permutation(self.num_blocks - 1)
        self.alloc = BlockAllocator(self.num_blocks, order=order)
        self.initial_lens = ctx0.copy()
        self.initial_blocks = [self.alloc.allocate(-(-int(c) // bs)) for c in ctx0]

        # draw the whole schedule now (host bookkeeping only). bookkeeping_seconds:
        # the host time of the iterations' scheduler work (finishes, joins, one
        # block table per step), the allocator's conservation check excluded
        lens = ctx0.copy()
        blocks = [list(b) for b in self.initial_blocks]
        self.schedule = []
        t_start, t_check = time.perf_counter(), 0.0
        for it in range(iterations):
            fin = np.nonzero(rng.random(batch) < p_finish)[0].tolist()
            freed, joins = [], []
            for b in fin:
                freed += self.alloc.free(blocks[b])
            for b in fin:
                plen = int(loguniform(rng, prompt_lo, prompt_hi, 1)[0])
                blocks[b] = self.alloc.allocate(-(-plen // bs))
                lens[b] = plen
                joins.append((b, plen))
            slots = np.empty(batch, dtype=np.int64)
            for b in range(batch):
                if lens[b] % bs == 0:               # current block full: take a new one
                    blocks[b] += self.alloc.allocate(1)
                slots[b] = token_rows(blocks[b], 1, bs, start=int(lens[b]))[0]
                lens[b] += 1
            tc = time.perf_counter()
            self.alloc.check()
            t_check += time.perf_counter() - tc
            self.schedule.append(dict(
                finished=fin, freed=freed, joins=joins, slots=slots,
                tables=pad_tables(blocks, self.max_blocks),
                lens=torch.from_numpy(lens.astype(np.int32).copy()),
                blocks=[list(b) for b in blocks]))
        self.bookkeeping_seconds = time.perf_counter() - t_start - t_check

    # -- tensors ---------------------------------------------------------------
    def initial_caches(self, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
        """The pool before iteration 0: owned token rows N(0,1), the rest NaN.
        Rows are drawn sequence by sequence and copied to ``device`` in chunks."""
        H, D, bs = self.Hkv, self.D, self.bs
        kc = nan_pool(self.num_blocks, bs, H, D).to(device)
        vc = nan_pool(self.num_blocks, bs, H, D).to(device)
        kf, vf = kc.view(-1, H, D), vc.view(-1, H, D)
        gk, gv = _torch_gen(self.seed, 11), _torch_gen(self.seed, 12)
        for b in range(self.B):
            n = int(self.initial_lens[b])
            rows = torch.from_numpy(token_rows(self.initial_blocks[b], n, bs)).to(device)
            kf[rows] = randn_bf16(gk, (n, H, D)).to(device)
            vf[rows] = randn_bf16(gv, (n, H, D)).to(device)
        return kc, vc

    def step(self, it: int) -> CBStep:
        s = self.schedule[it]
        H, D, bs = self.Hkv, self.D, self.bs
        g = _torch_gen(self.seed, 100 + it)
        fill_rows, nfill = [], 0
        for b, plen in s["joins"]:
            fill_rows.append(token_rows(s["blocks"][b], plen, bs))
            nfill += plen
        fill_slots = torch.from_numpy(np.concatenate(fill_rows) if fill_rows
                                      else np.zeros(0, dtype=np.int64))
        return CBStep(
            index=it, finished=list(s["finished"]), freed=list(s["freed"]),
            fill_slots=fill_slots, fill_k=randn_bf16(g, (nfill, H, D)),
            fill_v=randn_bf16(g, (nfill, H, D)),
            slot_mapping=torch.from_numpy(s["slots"].copy()),
            k_new=randn_bf16(g, (self.B, H, D)), v_new=randn_bf16(g, (self.B, H, D)),
            q=randn_bf16(g, (self.B, self.Hq, D)),
            block_tables=s["tables"], context_lens=s["lens"])


def kv_bytes_of_step(context_lens, num_kv_heads: int, head_dim: int,
                     bytes_per_value: int = 2) -> int:
    """Algorithmic KV bytes one decode step reads: each cached token's K and V
    row of every KV head exactly once (one layer)."""
    return int(np.asarray(context_lens, dtype=np.int64).sum()) * 2 * num_kv_heads * head_dim * bytes_per_value


def fp8_pool(case: DecodeCase, seed: int = 0) -> dict:
    """An e4m3 copy of a case's pool for the FP8 KV cache: per-KV-head scales
    drawn in [1/32, 3/64) (N(0,1) values stay far inside the +-448 range), codes
    by torch's float8_e4m3fn cast of value / scale (NaN-poisoned slots stay NaN)."""
    rng = np.random.Generator(np.random.PCG64(seed + 11_000))
    H = case.num_kv_heads
    ks = (1.0 / 32.0 * (1.0 + 0.5 * rng.random(H))).astype(np.float32)
    vs = (1.0 / 32.0 * (1.0 + 0.5 * rng.random(H))).astype(np.float32)

    def codes(pool, s):
        x = pool.float() / torch.from_numpy(s)[:, None]
        return x.to(torch.float8_e4m3fn).view(torch.uint8)

    return {"k_codes": codes(case.k_cache, ks), "v_codes": codes(case.v_cache, vs),
            "k_scale": torch.from_numpy(ks), "v_scale": torch.from_numpy(vs)}
