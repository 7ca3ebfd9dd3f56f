"""fp64 CPU oracle: paged-KV decode attention with grouped-query heads.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``). Plain NumPy, float64,
no blocking, fusion or reordering beyond what each definition states.

Data conventions (shared with the input generators, not with the kernels):

* bfloat16 tensors arrive as ``uint16`` bit patterns. bfloat16 is the upper
  half of an IEEE-754 binary32 word, so widening is exact.
* ``k_cache`` / ``v_cache``: ``[num_blocks, block_size, num_kv_heads, head_dim]``.
  The page "Text Generation Inference: Hugging Face's production-grade LLM
  inference server" (section "Under the Hood: PagedAttention", its simplified
  forward pass) stores K and V interleaved in one pool,
  ``[num_physical_blocks, block_size, 2, num_heads, head_dim]``, and says
  "num_heads" where the KV heads are meant. We keep K and V in two pools of
  the same per-token layout; the gather below is unchanged by that choice.
* ``block_tables``: ``[B, max_blocks]`` ints; ``context_lens``: ``[B]`` ints,
  the number of cached tokens each sequence attends over (after the append).
* ``q``: ``[B, num_q_heads, head_dim]``; query head ``h`` reads KV head
  ``h // G`` with ``G = num_q_heads // num_kv_heads`` (contiguous groups).
  The pages state grouped-query attention ("How to Speed Up LLM Inference:
  KV Cache to Production Serving", section "The KV cache: the memory problem
  that runs the show", item 3 "Shrink it by design"; "The inference request
  lifecycle", section "KV cache grows with the sum of cached tokens") but not
  which query heads share a KV head; contiguous groups are the plain reading.

parity: every function below is pinned in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# number formats and sizes
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (``uint16``) to float64, exactly."""
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError(f"bfloat16 data must be passed as uint16 bits, got {b.dtype}")
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int,
                       bytes_per_value: int) -> int:
    """Bytes of KV cache one token occupies across the whole model.

    The factor 2 is one K and one V vector per layer per KV head. Stated in
    "Text Generation Inference ..." (section "Production Pattern: KV Cache
    Math"), "How to Speed Up LLM Inference ..." (section "The KV cache: the
    memory problem that runs the show") and "The inference request lifecycle"
    (sections "KV cache grows with the sum of cached tokens" and "Work the GQA
    number before choosing concurrency").
    """
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_value


# ---------------------------------------------------------------------------
# KV append (slot write)
# ---------------------------------------------------------------------------

def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
              v_new: np.ndarray, slot_mapping) -> tuple[np.ndarray, np.ndarray]:
    """Return copies of the caches with each new token's K/V row written.

    Token ``t`` goes to flat slot ``slot_mapping[t]``: physical block
    ``slot // block_size``, offset ``slot % block_size``. This is the append
    of "Text Generation Inference ..." (section "Under the Hood:
    PagedAttention": a new token's KV pair goes into the current block, a new
    physical block being taken when it is full); which slot that is, is the
    block allocator's decision and arrives here as ``slot_mapping``.
    ``slot < 0`` marks a padded row and is skipped. A slot past the pool is
    an error. Bit patterns are copied unchanged.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    kv_append_inplace(kc, vc, k_new, v_new, slot_mapping)
    return kc, vc


def kv_append_inplace(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                      v_new: np.ndarray, slot_mapping) -> None:
    """:func:`kv_append` writing into the given caches instead of copies."""
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        if slot >= nb * bs:
            raise IndexError(f"slot {slot} outside a pool of {nb * bs} slots")
        k_cache[slot // bs, slot % bs] = k_new[t]
        v_cache[slot // bs, slot % bs] = v_new[t]


# ---------------------------------------------------------------------------
# block-table gather
# ---------------------------------------------------------------------------

def gather_sequence(cache: np.ndarray, block_table_row, ctx: int) -> np.ndarray:
    """Contiguous rows ``[ctx, H_kv, D]`` of one sequence's logical tokens.

    Logical token ``t`` lives in physical block ``block_table_row[t // bs]`` at
    offset ``t % bs`` ("Text Generation Inference ...", section "Under the
    Hood: PagedAttention": the block table maps logical block indices to
    physical blocks of a shared pool, like a page table). Positions at or past
    ``ctx`` in the last block are not part of the sequence.
    """
    bs = cache.shape[1]
    n_blocks = -(-ctx // bs)
    phys = np.asarray(block_table_row[:n_blocks], dtype=np.int64)
    blocks = cache[phys]                                   # [n_blocks, bs, H, D]
    return blocks.reshape((n_blocks * bs,) + cache.shape[2:])[:ctx]


def _group(q: np.ndarray, k_cache: np.ndarray) -> int:
    hq, hkv = q.shape[1], k_cache.shape[2]
    if hq % hkv:
        raise ValueError(f"{hq} query heads do not split into {hkv} KV heads")
    return hq // hkv


def _seq_list(B: int, seqs):
    return list(range(B)) if seqs is None else [int(s) for s in seqs]


# ---------------------------------------------------------------------------
# decode attention: the plain definition (two passes over the scores)
# ---------------------------------------------------------------------------

def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
           seqs=None) -> np.ndarray:
    """float64 decode attention output ``[len(seqs), H_q, D]``.

    For each sequence ``b`` and query head ``h``: gather the sequence's K and V
    rows, ``s = scale * K[:, h // G] @ q[b, h]``, ``out = softmax(s) @ V[:, h // G]``.
    Softmax runs over all ``context_lens[b]`` positions of the sequence (the
    page's simplified loop applies softmax to one score at a time, which is
    always 1; the whole-row softmax of "Under the Hood: Flash Attention" is the
    reading taken). ``context_lens[b] == 0`` gives zeros. ``seqs`` selects a
    subset of sequences (default: all).
    """
    G = _group(q, k_cache)
    rows = _seq_list(q.shape[0], seqs)
    hq, d = q.shape[1], q.shape[2]
    out = np.zeros((len(rows), hq, d), dtype=np.float64)
    for i, b in enumerate(rows):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_tables[b], ctx))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_tables[b], ctx))
        qb = bf16_bits_to_f64(q[b])
        for h in range(hq):
            kvh = h // G
            s = scale * (K[:, kvh, :] @ qb[h])
            p = np.exp(s - s.max())
            out[i, h] = (p @ V[:, kvh, :]) / p.sum()
    return out


# ---------------------------------------------------------------------------
# decode attention: the streaming (online-softmax) recurrence
# ---------------------------------------------------------------------------

def decode_online(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                  tile: int = 16, seqs=None) -> np.ndarray:
    """Same result as :func:`decode`, by the tiled recurrence of "Text
    Generation Inference ..." (section "Under the Hood: Flash Attention").

    One query row per head; the key/value tiles are ``tile`` consecutive
    logical tokens. Per tile: new running max ``m'`` = max of the old one and
    the tile's scores, ``P = exp(S - m')``, ``l = exp(m - m') * l + sum(P)``,
    ``O = exp(m - m') * O + P @ V``, ``m = m'``; at the end ``O / l``.
    """
    G = _group(q, k_cache)
    rows = _seq_list(q.shape[0], seqs)
    hq, d = q.shape[1], q.shape[2]
    out = np.zeros((len(rows), hq, d), dtype=np.float64)
    for i, b in enumerate(rows):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_tables[b], ctx))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_tables[b], ctx))
        qb = bf16_bits_to_f64(q[b])
        for h in range(hq):
            kvh = h // G
            m, l, O = -math.inf, 0.0, np.zeros(d)
            for j in range(0, ctx, tile):
                Kj, Vj = K[j:j + tile, kvh, :], V[j:j + tile, kvh, :]
                S = scale * (Kj @ qb[h])
                m_new = max(m, float(S.max()))
                P = np.exp(S - m_new)
                l = math.exp(m - m_new) * l + float(P.sum())
                O = math.exp(m - m_new) * O + P @ Vj
                m = m_new
            out[i, h] = O / l
    return out


# ---------------------------------------------------------------------------
# context split ("flash-decoding") partials and their log-sum-exp merge
# ---------------------------------------------------------------------------

def decode_split_partials(q, k_cache, v_cache, block_tables, context_lens,
                          scale: float, split_tokens: int, max_splits: int,
                          seqs=None):
    """Per-split partial results ``(part_out [n, H_q, S, D], part_lse [n, H_q, S])``.

    Split ``s`` of sequence ``b`` covers logical tokens
    ``[s * split_tokens, min((s + 1) * split_tokens, ctx_b))``. Its partial is
    the attention output over those tokens alone (normalised) and
    ``lse_s = log(sum_t exp(scale * q . k_t))`` in natural log. A split with
    no tokens has ``lse = -inf`` and a zero output. The pages do not describe
    splitting; this partial format rests on the rescaling algebra of "Under
    the Hood: Flash Attention" and is merged by :func:`lse_merge`.
    """
    G = _group(q, k_cache)
    rows = _seq_list(q.shape[0], seqs)
    hq, d = q.shape[1], q.shape[2]
    po = np.zeros((len(rows), hq, max_splits, d))
    pl = np.full((len(rows), hq, max_splits), -np.inf)
    for i, b in enumerate(rows):
        ctx = int(context_lens[b])
        if ctx > max_splits * split_tokens:
            raise ValueError("context longer than max_splits * split_tokens")
        if ctx == 0:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_tables[b], ctx))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_tables[b], ctx))
        qb = bf16_bits_to_f64(q[b])
        for h in range(hq):
            kvh = h // G
            s_all = scale * (K[:, kvh, :] @ qb[h])
            for s in range(max_splits):
                lo, hi = s * split_tokens, min((s + 1) * split_tokens, ctx)
                if lo >= hi:
                    continue
                x = s_all[lo:hi]
                mx = x.max()
                p = np.exp(x - mx)
                po[i, h, s] = (p @ V[lo:hi, kvh, :]) / p.sum()
                pl[i, h, s] = mx + math.log(p.sum())
    return po, pl


def lse_merge(part_out: np.ndarray, part_lse: np.ndarray) -> np.ndarray:
    """Merge split partials: ``M = max_s lse_s``, ``w_s = exp(lse_s - M)``,
    ``out = sum_s w_s O_s / sum_s w_s``. Splits with ``lse = -inf`` carry no
    tokens and are skipped; if every split is empty the output is zero."""
    n, hq, S, d = part_out.shape
    out = np.zeros((n, hq, d))
    for i in range(n):
        for h in range(hq):
            lse = part_lse[i, h]
            live = np.isfinite(lse)
            if not live.any():
                continue
            M = lse[live].max()
            w = np.exp(lse[live] - M)
            out[i, h] = (w @ part_out[i, h, live]) / w.sum()
    return out


# ---------------------------------------------------------------------------
# brute force in the pages' own loop structure (tiny inputs only)
# ---------------------------------------------------------------------------

def decode_pseudocode_loops(q, k_cache, v_cache, block_tables, context_lens,
                            scale: float) -> list:
    """Pure-Python scalar loops, following the structure of the simplified
    PagedAttention forward pass ("Text Generation Inference ...", section
    "Under the Hood: PagedAttention"): walk the block table, then the positions
    of each physical block, reading K and V at ``pool[physical_block][pos]``.

    Readings taken where that listing is silent or garbled: positions at or
    past the sequence length are skipped, and the softmax runs over all the
    sequence's scores (collected first, then normalised) instead of over one
    score. No NumPy vector arithmetic; returns nested lists ``[B][H_q][D]``.
    """
    B, hq, d = len(q), len(q[0]), len(q[0][0])
    nb, bs, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    G = hq // hkv

    def f(bits) -> float:
        return float(bf16_bits_to_f64(np.asarray([bits], dtype=np.uint16))[0])

    out = []
    for b in range(B):
        ctx = int(context_lens[b])
        per_head = []
        for h in range(hq):
            kvh = h // G
            scores, values = [], []
            pos_logical = 0
            for block_idx in range(len(block_tables[b])):
                if pos_logical >= ctx:
                    break
                physical_block = int(block_tables[b][block_idx])
                for pos in range(bs):
                    if pos_logical >= ctx:
                        break
                    dot = 0.0
                    for e in range(d):
                        dot += f(q[b][h][e]) * f(k_cache[physical_block][pos][kvh][e])
                    scores.append(scale * dot)
                    values.append([f(v_cache[physical_block][pos][kvh][e]) for e in range(d)])
                    pos_logical += 1
            if not scores:
                per_head.append([0.0] * d)
                continue
            mx = max(scores)
            w = [math.exp(s - mx) for s in scores]
            tot = sum(w)
            per_head.append([sum(w[t] * values[t][e] for t in range(len(w))) / tot
                             for e in range(d)])
        out.append(per_head)
    return out


# ---------------------------------------------------------------------------
# several query tokens per sequence (chunked prefill, speculative verification)
# ---------------------------------------------------------------------------
# "Text Generation Inference ...", section "Advanced Pattern: Chunked Prefill
# (TGI v3)": a prompt is processed in chunks interleaved with decode steps;
# "How to Speed Up LLM Inference ...", section "Speculative decoding: more
# than one token per weight-read": the target model checks the gamma drafted
# tokens plus one in a single pass. Either way a sequence brings q_len new
# query tokens, appended at the end of its context. Reading taken (the pages
# state no mask): the new tokens hold the last q_len positions of the context
# (after the append), and the token at position p attends to positions
# 0..p -- everything before it and itself, nothing after (causal).

def decode_multi(q_rows, k_cache, v_cache, block_tables, context_lens, q_start,
                 scale: float) -> np.ndarray:
    """float64 attention output ``[R, H_q, D]`` for packed query rows.

    ``q_rows`` holds bf16 bits ``[R, H_q, D]``: sequence ``b`` owns rows
    ``q_start[b] .. q_start[b+1]-1``, its ``n_b`` new tokens in order, and row
    ``q_start[b] + i`` sits at position ``p = context_lens[b] - n_b + i``. For
    each such row and query head ``h``: ``softmax(scale * K[0..p, h // G] q) @
    V[0..p, h // G]``. Rows with ``p < 0`` (more new tokens than context) are
    zero.
    """
    G = _group(q_rows, k_cache)
    R, hq, d = q_rows.shape
    out = np.zeros((R, hq, d), dtype=np.float64)
    for b in range(len(context_lens)):
        r0, r1 = int(q_start[b]), int(q_start[b + 1])
        n = r1 - r0
        ctx = int(context_lens[b])
        if n == 0 or ctx == 0:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_tables[b], ctx))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_tables[b], ctx))
        for i in range(n):
            pos = ctx - n + i
            if pos < 0:
                continue
            qi = bf16_bits_to_f64(q_rows[r0 + i])
            for h in range(hq):
                kvh = h // G
                s = scale * (K[:pos + 1, kvh, :] @ qi[h])
                w = np.exp(s - s.max())
                out[r0 + i, h] = (w @ V[:pos + 1, kvh, :]) / w.sum()
    return out


# ---------------------------------------------------------------------------
# FP8 (e4m3) KV cache
# ---------------------------------------------------------------------------
# "How to Speed Up LLM Inference: KV Cache to Production Serving" (section "The
# KV cache: the memory problem that runs the show": quantizing the cache itself
# to FP8 halves the bytes per token) and the FP8 row of "Text Generation
# Inference ..." (section "Production Pattern: KV Cache Math", 163,840 B/token)
# fix only the byte count. Readings taken: the OCP e4m3 format (1 sign bit,
# 4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is
# NaN, largest finite 448); one scale per KV head for K and one for V; a stored
# code is the round-to-nearest-even e4m3 value of x / scale computed in
# float32, saturated to +-448; a code reads back as value(code) * scale.

def e4m3_value(code: int) -> float:
    """The real number an e4m3 code stands for (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:                                   # subnormal: man/8 * 2^(1-7)
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0


def e4m3_encode(x) -> np.ndarray:
    """Round each float to the nearest e4m3 code, ties to the even code,
    saturating finite values beyond +-448 to +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.array([c for c in range(0x7F)], dtype=np.int64)      # 0x00 .. 0x7E, increasing
    vals = E4M3_TABLE[pos]
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(vals, a, side="left")                      # first value >= a
    hi = np.clip(hi, 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (pos[hi] % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, pos[hi], pos[lo])
    code = np.where(a == vals[hi], pos[hi], code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 codes (uint8)."""
    c = np.asarray(codes)
    if c.dtype != np.uint8:
        raise TypeError("e4m3 codes must be uint8")
    return E4M3_TABLE[c]


def quantize_rows_e4m3(rows_bf16_bits: np.ndarray, scale_per_head) -> np.ndarray:
    """e4m3 codes of bf16 rows [..., H_kv, D]: x / scale_h in float32, then
    e4m3_encode."""
    x = (np.asarray(rows_bf16_bits).astype(np.uint32) << np.uint32(16)).view(np.float32)
    s = np.asarray(scale_per_head, dtype=np.float32)[:, None]
    return e4m3_encode((x / s).astype(np.float32))


def kv_append_fp8_inplace(k_codes, v_codes, k_new_bits, v_new_bits, slot_mapping,
                          k_scale, v_scale) -> None:
    """The append into an e4m3 pool: quantize each new row, write it at its slot
    (slot < 0 skipped, a slot past the pool is an error)."""
    kq = quantize_rows_e4m3(k_new_bits, k_scale)
    vq = quantize_rows_e4m3(v_new_bits, v_scale)
    kv_append_inplace(k_codes, v_codes, kq, vq, slot_mapping)


def dequantize_pool(codes: np.ndarray, scale_per_head) -> np.ndarray:
    """float64 [NB, bs, H_kv, D] values of an e4m3 pool."""
    return e4m3_decode(codes) * np.asarray(scale_per_head, dtype=np.float64)[:, None]


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
               scale: float, seqs=None) -> np.ndarray:
    """:func:`decode` over an e4m3 pool: the K/V rows are read back as
    value(code) * scale of their head, then the same softmax attention."""
    G = _group(q, k_codes)
    rows = _seq_list(q.shape[0], seqs)
    hq, d = q.shape[1], q.shape[2]
    ks = np.asarray(k_scale, dtype=np.float64)
    vs = np.asarray(v_scale, dtype=np.float64)
    out = np.zeros((len(rows), hq, d), dtype=np.float64)
    for i, b in enumerate(rows):
        ctx = int(context_lens[b])
        if ctx == 0:
            continue
        K = e4m3_decode(gather_sequence(k_codes, block_tables[b], ctx)) * ks[:, None]
        V = e4m3_decode(gather_sequence(v_codes, block_tables[b], ctx)) * vs[:, None]
        qb = bf16_bits_to_f64(q[b])
        for h in range(hq):
            kvh = h // G
            s = scale * (K[:, kvh, :] @ qb[h])
            p = np.exp(s - s.max())
            out[i, h] = (p @ V[:, kvh, :]) / p.sum()
    return out


def decode_multi_fp8(q_rows, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                     q_start, scale: float) -> np.ndarray:
    """:func:`decode_multi` over an e4m3 pool: the K/V rows read back as
    value(code) * scale of their head, then for row q_start[b] + i (position
    p = context_lens[b] - n_b + i) and query head h, softmax(scale * K[0..p,
    h // G] q) @ V[0..p, h // G]; rows with p < 0 are zero."""
    G = _group(q_rows, k_codes)
    R, hq, d = q_rows.shape
    ks = np.asarray(k_scale, dtype=np.float64)
    vs = np.asarray(v_scale, dtype=np.float64)
    out = np.zeros((R, hq, d), dtype=np.float64)
    for b in range(len(context_lens)):
        r0, r1 = int(q_start[b]), int(q_start[b + 1])
        n = r1 - r0
        ctx = int(context_lens[b])
        if n == 0 or ctx == 0:
            continue
        K = e4m3_decode(gather_sequence(k_codes, block_tables[b], ctx)) * ks[:, None]
        V = e4m3_decode(gather_sequence(v_codes, block_tables[b], ctx)) * vs[:, None]
        for i in range(n):
            pos = ctx - n + i
            if pos < 0:
                continue
            qi = bf16_bits_to_f64(q_rows[r0 + i])
            for h in range(hq):
                kvh = h // G
                sc = scale * (K[:pos + 1, kvh, :] @ qi[h])
                w = np.exp(sc - sc.max())
                out[r0 + i, h] = (w @ V[:pos + 1, kvh, :]) / w.sum()
    return out

