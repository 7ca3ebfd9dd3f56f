"""Shared helpers for the GPU parity tests: move a seeded case to the device,
run the library through the C ABI, and compare with the fp64 oracle.

Tolerance for bf16 attention outputs against the fp64 oracle: max absolute
error <= 2e-2 and, per (sequence, query head) row, relative L2 error
<= 5e-3. The append and all indexing are compared bit for bit.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import paged_attention as pa
from paged_kv_cache_45_gb300 import workloads as wl

MAX_ABS = 2e-2
MAX_REL_L2 = 5e-3


def dev(case, device="cuda"):
    """Device copies of a case's tensors (caches before the append)."""
    d = dict(q=case.q.to(device), k_cache=case.k_cache.to(device),
             v_cache=case.v_cache.to(device), block_tables=case.block_tables.to(device),
             context_lens=case.context_lens.to(device))
    if case.k_new is not None:
        d.update(k_new=case.k_new.to(device), v_new=case.v_new.to(device),
                 slot_mapping=case.slot_mapping.to(device))
    return d


def oracle_caches(case):
    kc, vc = wl.bits(case.k_cache), wl.bits(case.v_cache)
    if case.k_new is None:
        return kc, vc
    return pa.kv_append(kc, vc, wl.bits(case.k_new), wl.bits(case.v_new),
                        case.slot_mapping.numpy())


def oracle_out(case, seqs=None, caches=None):
    kc, vc = caches if caches is not None else oracle_caches(case)
    return pa.decode(wl.bits(case.q), kc, vc, case.block_tables.numpy(),
                     case.context_lens.numpy(), case.scale, seqs=seqs)


def to_f64(out_bf16: torch.Tensor) -> np.ndarray:
    return out_bf16.float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    """(max abs error, max per-row relative L2 error); rows are the last axis."""
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    num = np.sqrt((diff ** 2).sum(-1))
    den = np.sqrt((ref ** 2).sum(-1))
    rel = np.where(den > 0, num / np.maximum(den, 1e-30), num)
    return max_abs, float(rel.max()) if rel.size else 0.0


def assert_close(got, ref, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    assert max_abs <= MAX_ABS and rel <= MAX_REL_L2, \
        f"{what}: max_abs={max_abs:.3e} (<= {MAX_ABS}), max_rel_l2={rel:.3e} (<= {MAX_REL_L2})"
    return max_abs, rel
