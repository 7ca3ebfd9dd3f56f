"""Thin ctypes binding of ``libpagedkv.so`` (declared in ``include/pagedkv.h``).

The functions carry the C names and only marshal arguments: they check that
tensors are CUDA, contiguous and of the declared dtype, pass their
``data_ptr()`` and the current torch stream, and raise ``PagedKVError`` on a
non-OK status. Every step of the computation runs in the library's kernels.
PyTorch supplies device memory and streams.

Importing this module loads the library and raises ``ImportError`` if it has
not been built (``python -m paged_kv_cache_45_gb300.build``): there is no
fallback of any kind.
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing; build it with "
                      "`python -m paged_kv_cache_45_gb300.build` (needs nvcc)")
_lib = ctypes.CDLL(_LIB_PATH)

_p, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)

_SIGS = {
    "pa_kv_append": (_i32, [_p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _p]),
    "pa_decode": (_i32, [_p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
                         _i32, _i32, _p, _p, _p, _p]),
    "pa_decode_splitk_reduce": (_i32, [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, _p, _p]),
    "pa_decode_balanced": (_i32, [_p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32,
                                  _f32, _p, _sz, _p, _p]),
    "pa_decode_balanced_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "pa_append_decode": (_i32, [_p, _p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32,
                                _i32, _i32, _f32, _p, _sz, _p, _p]),
    "pa_kv_append_fp8": (_i32, [_p, _p, _p, _i32, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _p]),
    "pa_decode_balanced_fp8": (_i32, [_p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32,
                                      _i32, _i32, _f32, _p, _sz, _p, _p]),
    "pa_append_decode_fp8": (_i32, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i32, _p, _i32, _i32,
                                    _i32, _i32, _i32, _i32, _f32, _p, _sz, _p, _p]),
    "pa_decode_balanced_static": (_i32, [_p, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32,
                                         _i32, _f32, _p, _p]),
    "pa_decode_num_splits": (_i32, [_i32, _i32]),
    "pa_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "pa_kv_bytes_per_token": (_i64, [_i32, _i32, _i32, _i32]),
    "pa_last_device_error": (_i32, [ctypes.POINTER(_i32)]),
    "pa_selftest_wait_timeout": (_i32, [_i32, _p]),
    "pa_decode_multi": (_i32, [_p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32,
                               _i32, _i32, _f32, _i32, _i32, _p, _p, _p, _p, _p]),
    "pa_decode_multi_balanced": (_i32, [_p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32,
                                        _i32, _i32, _i32, _i32, _f32, _p, _sz, _p, _p]),
    "pa_decode_multi_balanced_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "pa_decode_multi_fp8": (_i32, [_p, _p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _i32, _i32,
                                   _i32, _i32, _i32, _i32, _f32, _i32, _i32, _p, _p, _p, _p, _p]),
    "pa_prefix_cache_create": (_i32, [_i32, _i32, _p]),
    "pa_prefix_cache_destroy": (None, [_p]),
    "pa_prefix_admit": (_i32, [_p, _p, _i32, _p, _p]),
    "pa_prefix_write_slots": (_i32, [_p, _i64, _i32, _i32, _p, _p, _p, _i32, _p]),
    "pa_prefix_append_tokens": (_i32, [_p, _p, _i32, _p, _p, _p, _i32, _p, _p]),
    "pa_prefix_fork": (_i32, [_p, _i64, _p]),
    "pa_prefix_fork_batch": (_i32, [_p, _p, _i32, _p]),
    "pa_prefix_discard": (_i32, [_p, _p, _i32]),
    "pa_prefix_release": (_i32, [_p, _i64, _p, _i32]),
    "pa_prefix_table": (_i32, [_p, _i64, _p, _i32, _p, _p]),
    "pa_prefix_tables": (_i32, [_p, _p, _i32, _p, _i32, _p]),
    "pa_prefix_stats": (_i32, [_p, _p, _p, _p]),
    "pa_prefix_evictable": (_i32, [_p, _p]),
    "pa_copy_blocks": (_i32, [_p, _p, _p, _p, _i32, _i32, _i64, _p]),
    "pa_status_str": (ctypes.c_char_p, [_i32]),
    "pa_version": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype, _fn.argtypes = _res, _args

EXPORTS = tuple(_SIGS)
LIBRARY_PATH = _LIB_PATH


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {pa_status_str(status)} ({status})")
        self.status = status


def pa_status_str(status: int) -> str:
    return _lib.pa_status_str(int(status)).decode()


def pa_version() -> str:
    return _lib.pa_version().decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise PagedKVError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _t(x: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return x.data_ptr()


def _opt(x, dtype, name):
    return None if x is None else _t(x, dtype, name)


# ---------------------------------------------------------------------------
# the three entry points of the hot path
# ---------------------------------------------------------------------------

def pa_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Scatter ``k_new``/``v_new`` [T, Hkv, D] into the caches [NB, bs, Hkv, D]
    at ``slot_mapping`` [T] (int64; negative = skip)."""
    nb, bs, hkv, d = k_cache.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [T, num_kv_heads, head_dim] matching the caches")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or slot_mapping.numel() != T:
        raise ValueError("cache or slot_mapping shape mismatch")
    _check("pa_kv_append", _lib.pa_kv_append(
        _t(k_new, torch.bfloat16, "k_new"), _t(v_new, torch.bfloat16, "v_new"),
        _t(slot_mapping, torch.int64, "slot_mapping"), T,
        _t(k_cache, torch.bfloat16, "k_cache"), _t(v_cache, torch.bfloat16, "v_cache"),
        nb, bs, hkv, d, _stream(stream)))


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
              split_tokens: int = 0, max_splits: int = 0, part_out=None, part_lse=None,
              stream=None) -> None:
    """Paged decode attention into ``out`` [B, Hq, D] bf16 (or, with
    ``split_tokens > 0``, into the fp32 partials ``part_out``/``part_lse``)."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(out.shape) != (B, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    if context_lens.numel() != B:
        raise ValueError("context_lens must have one entry per sequence")
    _check("pa_decode", _lib.pa_decode(
        _t(q, torch.bfloat16, "q"), _t(k_cache, torch.bfloat16, "k_cache"),
        _t(v_cache, torch.bfloat16, "v_cache"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"), B, hq, hkv, d,
        bs, nb, float(scale), int(split_tokens), int(max_splits),
        _opt(part_out, torch.float32, "part_out"), _opt(part_lse, torch.float32, "part_lse"),
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def pa_decode_splitk_reduce(part_out, part_lse, context_lens, split_tokens: int, out,
                            stream=None) -> None:
    """Merge ``part_out`` [B, Hq, S, D] / ``part_lse`` [B, Hq, S] into ``out``."""
    B, hq, S, d = part_out.shape
    if tuple(part_lse.shape) != (B, hq, S) or tuple(out.shape) != (B, hq, d):
        raise ValueError("partial / output shape mismatch")
    _check("pa_decode_splitk_reduce", _lib.pa_decode_splitk_reduce(
        _t(part_out, torch.float32, "part_out"), _t(part_lse, torch.float32, "part_lse"),
        _t(context_lens, torch.int32, "context_lens"), B, hq, d, int(split_tokens), S,
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def pa_decode_multi(q, k_cache, v_cache, block_tables, context_lens, q_start, max_q_len: int,
                    scale: float, out, split_tokens: int = 0, max_splits: int = 0,
                    part_out=None, part_lse=None, row_lens=None, stream=None) -> None:
    """Causal attention for packed query rows ``q`` [R, Hq, D] (sequence b owns
    rows ``q_start[b]:q_start[b+1]``, its newest tokens) into ``out`` [R, Hq, D]
    (or, with ``split_tokens > 0``, into the partials and ``row_lens``)."""
    R, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    B = context_lens.numel()
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(out.shape) != (R, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    if q_start.numel() != B + 1:
        raise ValueError("q_start must have num_seqs + 1 entries")
    _check("pa_decode_multi", _lib.pa_decode_multi(
        _t(q, torch.bfloat16, "q"), _t(k_cache, torch.bfloat16, "k_cache"),
        _t(v_cache, torch.bfloat16, "v_cache"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"),
        _t(q_start, torch.int32, "q_start"), B, R, int(max_q_len), hq, hkv, d, bs, nb,
        float(scale), int(split_tokens), int(max_splits),
        _opt(part_out, torch.float32, "part_out"), _opt(part_lse, torch.float32, "part_lse"),
        _opt(row_lens, torch.int32, "row_lens"), _t(out, torch.bfloat16, "out"),
        _stream(stream)))


def pa_decode_multi_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                        q_start, max_q_len: int, scale: float, out, split_tokens: int = 0,
                        max_splits: int = 0, part_out=None, part_lse=None, row_lens=None,
                        stream=None) -> None:
    """pa_decode_multi over an e4m3 pool (uint8 codes, per-KV-head fp32 scales)."""
    R, hq, d = q.shape
    nb, bs, hkv, d2 = k_codes.shape
    B = context_lens.numel()
    if d2 != d or tuple(v_codes.shape) != tuple(k_codes.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(out.shape) != (R, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    if q_start.numel() != B + 1 or k_scale.numel() != hkv or v_scale.numel() != hkv:
        raise ValueError("q_start / scale sizes do not match")
    _check("pa_decode_multi_fp8", _lib.pa_decode_multi_fp8(
        _t(q, torch.bfloat16, "q"), _t(k_codes, torch.uint8, "k_codes"),
        _t(v_codes, torch.uint8, "v_codes"), _t(k_scale, torch.float32, "k_scale"),
        _t(v_scale, torch.float32, "v_scale"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"),
        _t(q_start, torch.int32, "q_start"), B, R, int(max_q_len), hq, hkv, d, bs, nb,
        float(scale), int(split_tokens), int(max_splits),
        _opt(part_out, torch.float32, "part_out"), _opt(part_lse, torch.float32, "part_lse"),
        _opt(row_lens, torch.int32, "row_lens"), _t(out, torch.bfloat16, "out"),
        _stream(stream)))


def pa_decode_multi_balanced(q, k_cache, v_cache, block_tables, context_lens, q_start,
                             max_q_len: int, scale: float, workspace, out, stream=None) -> None:
    """pa_decode_multi on the balanced persistent schedule; ``workspace`` a
    zero-filled uint8 CUDA tensor of ``pa_decode_multi_balanced_workspace_bytes``."""
    R, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    B = context_lens.numel()
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(out.shape) != (R, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    if q_start.numel() != B + 1:
        raise ValueError("q_start must have num_seqs + 1 entries")
    _check("pa_decode_multi_balanced", _lib.pa_decode_multi_balanced(
        _t(q, torch.bfloat16, "q"), _t(k_cache, torch.bfloat16, "k_cache"),
        _t(v_cache, torch.bfloat16, "v_cache"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"),
        _t(q_start, torch.int32, "q_start"), B, R, int(max_q_len), hq, hkv, d, bs, nb,
        float(scale), _t(workspace, torch.uint8, "workspace"), workspace.numel(),
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def pa_decode_multi_balanced_workspace_bytes(num_seqs: int, num_kv_heads: int,
                                             head_dim: int) -> int:
    return int(_lib.pa_decode_multi_balanced_workspace_bytes(int(num_seqs), int(num_kv_heads),
                                                             int(head_dim)))


BALANCED_MULTI = -1


def decode_multi(q, k_cache, v_cache, block_tables, context_lens, q_start, max_q_len: int,
                 scale: float, split_tokens: int = 0, max_context: int | None = None,
                 out=None, stream=None):
    """pa_decode_multi with its split-mode buffers and the reduce (or, with
    ``split_tokens == BALANCED_MULTI``, pa_decode_multi_balanced); returns out."""
    R, hq, d = q.shape
    if out is None:
        out = torch.empty((R, hq, d), dtype=torch.bfloat16, device=q.device)
    if split_tokens == BALANCED_MULTI:
        ws = torch.zeros(pa_decode_multi_balanced_workspace_bytes(
            context_lens.numel(), k_cache.shape[2], d), dtype=torch.uint8, device=q.device)
        pa_decode_multi_balanced(q, k_cache, v_cache, block_tables, context_lens, q_start,
                                 max_q_len, scale, ws, out, stream=stream)
        return out
    if split_tokens <= 0:
        pa_decode_multi(q, k_cache, v_cache, block_tables, context_lens, q_start, max_q_len,
                        scale, out, stream=stream)
        return out
    if max_context is None:
        max_context = int(block_tables.shape[1]) * int(k_cache.shape[1])
    S = pa_decode_num_splits(max_context, split_tokens)
    part_out = torch.empty((R, hq, S, d), dtype=torch.float32, device=q.device)
    part_lse = torch.empty((R, hq, S), dtype=torch.float32, device=q.device)
    row_lens = torch.empty(R, dtype=torch.int32, device=q.device)
    pa_decode_multi(q, k_cache, v_cache, block_tables, context_lens, q_start, max_q_len, scale,
                    out, split_tokens, S, part_out, part_lse, row_lens, stream=stream)
    pa_decode_splitk_reduce(part_out, part_lse, row_lens, split_tokens, out, stream=stream)
    return out


def decode_multi_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                     q_start, max_q_len: int, scale: float, split_tokens: int = 0,
                     max_context: int | None = None, out=None, stream=None):
    """pa_decode_multi_fp8 with its split-mode buffers and the reduce; returns out."""
    R, hq, d = q.shape
    if out is None:
        out = torch.empty((R, hq, d), dtype=torch.bfloat16, device=q.device)
    if split_tokens <= 0:
        pa_decode_multi_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                            q_start, max_q_len, scale, out, stream=stream)
        return out
    if max_context is None:
        max_context = int(block_tables.shape[1]) * int(k_codes.shape[1])
    S = pa_decode_num_splits(max_context, split_tokens)
    part_out = torch.empty((R, hq, S, d), dtype=torch.float32, device=q.device)
    part_lse = torch.empty((R, hq, S), dtype=torch.float32, device=q.device)
    row_lens = torch.empty(R, dtype=torch.int32, device=q.device)
    pa_decode_multi_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens,
                        q_start, max_q_len, scale, out, split_tokens, S, part_out, part_lse,
                        row_lens, stream=stream)
    pa_decode_splitk_reduce(part_out, part_lse, row_lens, split_tokens, out, stream=stream)
    return out


def pa_decode_balanced(q, k_cache, v_cache, block_tables, context_lens, scale: float, workspace,
                       out, stream=None) -> None:
    """Work-balanced persistent decode into ``out`` [B, Hq, D] bf16 in one launch.
    ``workspace``: a zero-filled uint8 CUDA tensor of at least
    ``pa_decode_balanced_workspace_bytes(B, Hkv, D)`` bytes (left reusable)."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(out.shape) != (B, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    if context_lens.numel() != B:
        raise ValueError("context_lens must have one entry per sequence")
    _check("pa_decode_balanced", _lib.pa_decode_balanced(
        _t(q, torch.bfloat16, "q"), _t(k_cache, torch.bfloat16, "k_cache"),
        _t(v_cache, torch.bfloat16, "v_cache"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"), B, hq, hkv, d,
        bs, nb, float(scale), _t(workspace, torch.uint8, "workspace"), workspace.numel(),
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def pa_append_decode(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                     context_lens, scale: float, workspace, out, stream=None) -> None:
    """One step in one launch: append each sequence's new K/V row at its slot
    (the slot of its last logical token) and decode, as pa_kv_append followed
    by pa_decode_balanced. ``workspace`` as for pa_decode_balanced."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(k_new.shape) != (B, hkv, d) or tuple(v_new.shape) != (B, hkv, d):
        raise ValueError("k_new/v_new must be [num_seqs, num_kv_heads, head_dim]")
    if slot_mapping.numel() != B or context_lens.numel() != B:
        raise ValueError("slot_mapping and context_lens need one entry per sequence")
    if tuple(out.shape) != (B, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    _check("pa_append_decode", _lib.pa_append_decode(
        _t(q, torch.bfloat16, "q"), _t(k_new, torch.bfloat16, "k_new"),
        _t(v_new, torch.bfloat16, "v_new"), _t(slot_mapping, torch.int64, "slot_mapping"),
        _t(k_cache, torch.bfloat16, "k_cache"), _t(v_cache, torch.bfloat16, "v_cache"),
        _t(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
        _t(context_lens, torch.int32, "context_lens"), B, hq, hkv, d, bs, nb, float(scale),
        _t(workspace, torch.uint8, "workspace"), workspace.numel(),
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def _fp8_shapes(k_cache, v_cache, k_scale, v_scale):
    nb, bs, hkv, d = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache shapes differ")
    if k_scale.numel() != hkv or v_scale.numel() != hkv:
        raise ValueError("k_scale/v_scale need one entry per KV head")
    return nb, bs, hkv, d


def pa_kv_append_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                     stream=None) -> None:
    """Quantize ``k_new``/``v_new`` [T, Hkv, D] bf16 to e4m3 codes (x / scale of
    the head) at ``slot_mapping`` of the uint8 caches [NB, bs, Hkv, D]."""
    nb, bs, hkv, d = _fp8_shapes(k_cache, v_cache, k_scale, v_scale)
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, hkv, d) or tuple(v_new.shape) != (T, hkv, d):
        raise ValueError("k_new/v_new must be [T, num_kv_heads, head_dim]")
    if slot_mapping.numel() != T:
        raise ValueError("slot_mapping needs one entry per token")
    _check("pa_kv_append_fp8", _lib.pa_kv_append_fp8(
        _t(k_new, torch.bfloat16, "k_new"), _t(v_new, torch.bfloat16, "v_new"),
        _t(slot_mapping, torch.int64, "slot_mapping"), T, _t(k_cache, torch.uint8, "k_cache"),
        _t(v_cache, torch.uint8, "v_cache"), _t(k_scale, torch.float32, "k_scale"),
        _t(v_scale, torch.float32, "v_scale"), nb, bs, hkv, d, _stream(stream)))


def pa_decode_balanced_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                           scale: float, workspace, out, stream=None) -> None:
    """pa_decode_balanced over uint8 e4m3 caches with per-KV-head scales."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = _fp8_shapes(k_cache, v_cache, k_scale, v_scale)
    if d2 != d or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B:
        raise ValueError("q / out / cache / block_tables shapes do not match")
    _check("pa_decode_balanced_fp8", _lib.pa_decode_balanced_fp8(
        _t(q, torch.bfloat16, "q"), _t(k_cache, torch.uint8, "k_cache"),
        _t(v_cache, torch.uint8, "v_cache"), _t(k_scale, torch.float32, "k_scale"),
        _t(v_scale, torch.float32, "v_scale"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"), B, hq, hkv, d,
        bs, nb, float(scale), _t(workspace, torch.uint8, "workspace"), workspace.numel(),
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def pa_append_decode_fp8(q, k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                         block_tables, context_lens, scale: float, workspace, out,
                         stream=None) -> None:
    """pa_append_decode over uint8 e4m3 caches: quantize the new rows at their
    slots and decode, one launch."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = _fp8_shapes(k_cache, v_cache, k_scale, v_scale)
    if d2 != d or tuple(out.shape) != (B, hq, d) or block_tables.shape[0] != B:
        raise ValueError("q / out / cache / block_tables shapes do not match")
    if tuple(k_new.shape) != (B, hkv, d) or tuple(v_new.shape) != (B, hkv, d):
        raise ValueError("k_new/v_new must be [num_seqs, num_kv_heads, head_dim]")
    _check("pa_append_decode_fp8", _lib.pa_append_decode_fp8(
        _t(q, torch.bfloat16, "q"), _t(k_new, torch.bfloat16, "k_new"),
        _t(v_new, torch.bfloat16, "v_new"), _t(slot_mapping, torch.int64, "slot_mapping"),
        _t(k_cache, torch.uint8, "k_cache"), _t(v_cache, torch.uint8, "v_cache"),
        _t(k_scale, torch.float32, "k_scale"), _t(v_scale, torch.float32, "v_scale"),
        _t(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
        _t(context_lens, torch.int32, "context_lens"), B, hq, hkv, d, bs, nb, float(scale),
        _t(workspace, torch.uint8, "workspace"), workspace.numel(),
        _t(out, torch.bfloat16, "out"), _stream(stream)))


def pa_decode_balanced_static(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                              out, stream=None) -> None:
    """``pa_decode_balanced`` for callers that cannot allocate device memory:
    no workspace argument, the library's built-in 6 MiB device array serves as
    scratch. Calls on one device share that array, so calls whose kernels may
    overlap on the GPU must not be issued; the first call on a device should
    come before any stream capture (it looks the array's address up)."""
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match q")
    if tuple(out.shape) != (B, hq, d) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("out / block_tables shape mismatch")
    if context_lens.numel() != B:
        raise ValueError("context_lens must have one entry per sequence")
    _check("pa_decode_balanced_static", _lib.pa_decode_balanced_static(
        _t(q, torch.bfloat16, "q"), _t(k_cache, torch.bfloat16, "k_cache"),
        _t(v_cache, torch.bfloat16, "v_cache"), _t(block_tables, torch.int32, "block_tables"),
        int(block_tables.shape[1]), _t(context_lens, torch.int32, "context_lens"), B, hq, hkv, d,
        bs, nb, float(scale), _t(out, torch.bfloat16, "out"), _stream(stream)))


# ---------------------------------------------------------------------------
# sizes and diagnostics
# ---------------------------------------------------------------------------

def pa_decode_balanced_workspace_bytes(num_seqs: int, num_kv_heads: int, head_dim: int) -> int:
    return int(_lib.pa_decode_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim))


def pa_decode_num_splits(max_context: int, split_tokens: int) -> int:
    return int(_lib.pa_decode_num_splits(int(max_context), int(split_tokens)))


def pa_decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int,
                              max_splits: int) -> int:
    return int(_lib.pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_splits))


def pa_kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                          bytes_per_value: int) -> int:
    return int(_lib.pa_kv_bytes_per_token(num_layers, num_kv_heads, head_dim, bytes_per_value))


def pa_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait nobody completes runs out
    after ``limit_us``); pa_last_device_error() then returns bit 8."""
    _check("pa_selftest_wait_timeout", _lib.pa_selftest_wait_timeout(int(limit_us), _stream(stream)))


def pa_last_device_error() -> int:
    """Read and clear the device error word (synchronises); 0 means none."""
    code = _i32(0)
    st = _lib.pa_last_device_error(ctypes.byref(code))
    if st not in (0, -5):
        raise PagedKVError("pa_last_device_error", st)
    return int(code.value)


# ---------------------------------------------------------------------------
# convenience: one decode call with library-sized buffers
# ---------------------------------------------------------------------------

BALANCED = -1  # schedule selector: work-balanced persistent decode (pa_decode_balanced)


class DecodeWorkspace:
    """Output plus split partial buffers (``split_tokens > 0``) or the zero-filled
    balanced-schedule workspace (``split_tokens == BALANCED``) for repeated decode
    calls of one shape."""

    def __init__(self, num_seqs: int, num_q_heads: int, head_dim: int, split_tokens: int = 0,
                 max_context: int = 0, device="cuda", num_kv_heads: int | None = None):
        self.balanced = split_tokens == BALANCED
        self.scratch = None
        if self.balanced:
            if num_kv_heads is None:
                raise ValueError("the balanced schedule needs num_kv_heads")
            with torch.cuda.device(torch.device(device)):
                n = pa_decode_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim)
            self.scratch = torch.zeros(n, dtype=torch.uint8, device=device)
            split_tokens = 0
        self.split_tokens = int(split_tokens)
        self.max_splits = pa_decode_num_splits(max_context, split_tokens) if split_tokens else 0
        self.out = torch.empty((num_seqs, num_q_heads, head_dim), dtype=torch.bfloat16,
                               device=device)
        if self.split_tokens:
            self.part_out = torch.empty((num_seqs, num_q_heads, self.max_splits, head_dim),
                                        dtype=torch.float32, device=device)
            self.part_lse = torch.empty((num_seqs, num_q_heads, self.max_splits),
                                        dtype=torch.float32, device=device)
        else:
            self.part_out = self.part_lse = None


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
           ws: DecodeWorkspace | None = None, split_tokens: int = 0, max_context: int | None = None,
           stream=None) -> torch.Tensor:
    """``pa_decode`` (+ ``pa_decode_splitk_reduce`` when split), or
    ``pa_decode_balanced`` when ``split_tokens == BALANCED``, into a workspace;
    returns the bf16 output [B, Hq, D]."""
    B, hq, d = q.shape
    if ws is None:
        if split_tokens > 0 and max_context is None:
            max_context = int(block_tables.shape[1]) * int(k_cache.shape[1])
        ws = DecodeWorkspace(B, hq, d, split_tokens, max_context or 0, q.device,
                             num_kv_heads=int(k_cache.shape[2]))
    if ws.balanced:
        pa_decode_balanced(q, k_cache, v_cache, block_tables, context_lens, scale, ws.scratch,
                           ws.out, stream)
        return ws.out
    pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, ws.out, ws.split_tokens,
              ws.max_splits, ws.part_out, ws.part_lse, stream)
    if ws.split_tokens:
        pa_decode_splitk_reduce(ws.part_out, ws.part_lse, context_lens, ws.split_tokens, ws.out,
                                stream)
    return ws.out


# ---------------------------------------------------------------------------
# launch planning (host side)
# ---------------------------------------------------------------------------

def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


def plan_split(context_lens_host, num_kv_heads: int, sms: int = 152, blocks_per_sm: int = 16,
               lo: int = 256, hi: int = 8192) -> int:
    """Pick ``split_tokens`` for a batch whose lengths the host scheduler knows.

    Aims at about ``blocks_per_sm`` thread blocks' worth of KV per SM so the
    last wave's blocks are short next to the whole step (the tail), with
    powers of two in [lo, hi]. Returns 0 (no split, no reduce) when no
    sequence is longer than the chosen split.
    """
    import numpy as np
    lens = np.asarray(context_lens_host, dtype=np.int64)
    if lens.size == 0 or lens.max() <= 0:
        return 0
    per_block = lens.sum() * num_kv_heads / (sms * blocks_per_sm)
    split = lo
    while split < per_block and split < hi:
        split *= 2
    return 0 if lens.max() <= split else int(split)


# ---------------------------------------------------------------------------
# prefix cache (host) and copy-on-write (device)
# ---------------------------------------------------------------------------

PA_ERR_CAPACITY = -6


class CapacityError(PagedKVError):
    """The pool has no free or evictable block for the call (nothing changed)."""


def _host_i32(values):
    import numpy as np
    a = np.ascontiguousarray(np.asarray(values, dtype=np.int32))
    return a, a.ctypes.data


class PrefixCache:
    """Host block pool with a radix prefix cache and copy-on-write
    (``pa_prefix_*``). Methods mirror the C calls; copies come back as
    (src, dst) block pairs for :func:`pa_copy_blocks`."""

    def __init__(self, num_blocks: int, block_size: int):
        h = ctypes.c_void_p()
        _check("pa_prefix_cache_create",
               _lib.pa_prefix_cache_create(int(num_blocks), int(block_size), ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            _lib.pa_prefix_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _status(fn, st):
        if st == PA_ERR_CAPACITY:
            raise CapacityError(fn, st)
        _check(fn, st)

    def admit(self, tokens):
        arr, ptr = _host_i32(tokens)
        sid, cached = _i64(), _i32()
        self._status("pa_prefix_admit", _lib.pa_prefix_admit(
            self._h, ptr, len(arr), ctypes.byref(sid), ctypes.byref(cached)))
        return sid.value, cached.value

    def write_slots(self, seq_id, p0, p1):
        """Slots of positions [p0, p1) (int64 array) and the (src, dst) block
        copies to make first."""
        import numpy as np
        n = max(p1 - p0, 0)
        slots = np.empty(max(n, 1), dtype=np.int64)             # [0, n) is written
        nb = (p1 - 1) // self.block_size - p0 // self.block_size + 1 if n else 0
        src = np.zeros(max(nb, 1), dtype=np.int32)
        dst = np.zeros(max(nb, 1), dtype=np.int32)
        nc = _i32()
        self._status("pa_prefix_write_slots", _lib.pa_prefix_write_slots(
            self._h, int(seq_id), int(p0), int(p1), slots.ctypes.data, src.ctypes.data,
            dst.ctypes.data, len(src), ctypes.byref(nc)))
        k = nc.value
        return slots[:n], list(zip(src[:k].tolist(), dst[:k].tolist()))

    def append_tokens(self, seq_ids):
        """One decode position per sequence: (slots int64 array, copies, done)."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = len(ids)
        slots = np.zeros(max(n, 1), dtype=np.int64)
        src = np.zeros(max(n, 1), dtype=np.int32)
        dst = np.zeros(max(n, 1), dtype=np.int32)
        nc, done = _i32(), _i32()
        st = _lib.pa_prefix_append_tokens(self._h, ids.ctypes.data, n, slots.ctypes.data,
                                          src.ctypes.data, dst.ctypes.data, len(src),
                                          ctypes.byref(nc), ctypes.byref(done))
        copies = (src[:nc.value].copy(), dst[:nc.value].copy())
        if st == PA_ERR_CAPACITY:
            err = CapacityError("pa_prefix_append_tokens", st)
            err.done, err.slots, err.copies = done.value, slots[:done.value], copies
            raise err
        _check("pa_prefix_append_tokens", st)
        return slots[:n], copies

    def fork(self, seq_id):
        child = _i64()
        self._status("pa_prefix_fork", _lib.pa_prefix_fork(self._h, int(seq_id),
                                                           ctypes.byref(child)))
        return child.value

    def fork_batch(self, seq_ids):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        out = np.zeros(max(len(ids), 1), dtype=np.int64)
        self._status("pa_prefix_fork_batch", _lib.pa_prefix_fork_batch(
            self._h, ids.ctypes.data, len(ids), out.ctypes.data))
        return out[:len(ids)]

    def discard(self, seq_ids):
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        self._status("pa_prefix_discard", _lib.pa_prefix_discard(self._h, ids.ctypes.data,
                                                                 len(ids)))

    def release(self, seq_id, tokens):
        arr, ptr = _host_i32(tokens)
        self._status("pa_prefix_release", _lib.pa_prefix_release(self._h, int(seq_id), ptr,
                                                                 len(arr)))

    def table(self, seq_id):
        import numpy as np
        cap = self.num_blocks
        buf = np.zeros(cap, dtype=np.int32)
        nb, nt = _i32(), _i32()
        self._status("pa_prefix_table", _lib.pa_prefix_table(
            self._h, int(seq_id), buf.ctypes.data, cap, ctypes.byref(nb), ctypes.byref(nt)))
        return buf[:nb.value].tolist()

    def tables(self, seq_ids, max_blocks):
        """(block_tables int32 [n, max_blocks], context_lens int32 [n]) as numpy."""
        import numpy as np
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        t = np.empty((len(ids), max_blocks), dtype=np.int32)    # every entry is written
        lens = np.empty(len(ids), dtype=np.int32)
        self._status("pa_prefix_tables", _lib.pa_prefix_tables(
            self._h, ids.ctypes.data, len(ids), t.ctypes.data, int(max_blocks),
            lens.ctypes.data))
        return t, lens

    def stats(self):
        f, c, u = _i32(), _i32(), _i32()
        _check("pa_prefix_stats", _lib.pa_prefix_stats(self._h, ctypes.byref(f), ctypes.byref(c),
                                                       ctypes.byref(u)))
        return f.value, c.value, u.value

    def evictable(self) -> int:
        """Blocks eviction could free now (cached, unreferenced, nothing
        referenced after them on their prefix path)."""
        e = _i32()
        _check("pa_prefix_evictable", _lib.pa_prefix_evictable(self._h, ctypes.byref(e)))
        return e.value


def pa_copy_blocks(k_cache, v_cache, src, dst, stream=None) -> None:
    """Block dst[i] of both caches becomes a copy of block src[i] (device int32)."""
    if tuple(k_cache.shape) != tuple(v_cache.shape) or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must match")
    if src.numel() != dst.numel():
        raise ValueError("src and dst must have the same length")
    n = src.numel()
    if n == 0:
        return
    nb = k_cache.shape[0]
    block_bytes = k_cache.numel() // max(nb, 1) * k_cache.element_size()
    _check("pa_copy_blocks", _lib.pa_copy_blocks(
        _t(k_cache, k_cache.dtype, "k_cache"), _t(v_cache, v_cache.dtype, "v_cache"),
        _t(src, torch.int32, "src"), _t(dst, torch.int32, "dst"), n, nb, block_bytes,
        _stream(stream)))
