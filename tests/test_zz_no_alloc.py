"""pa_decode_balanced_static: the decode entry point for callers that cannot
allocate device memory at the call site (an engine that has reserved its free
HBM for the KV block pool, a plug-in without an allocator). It uses the
library's built-in scratch array instead of a workspace.

Checked through the C ABI on two calls in a row with different batches, so the
second call runs on whatever the first left in the shared array: against
pa_decode_balanced (the workspace entry point) and against the fp64 oracle.
Tolerance: the parity bar of the other tests (max abs <= 2e-2, per-row
relative L2 <= 5e-3). A shape whose scratch exceeds the array's 6 MiB must be
refused with PA_ERR_WORKSPACE before anything is written.

This file is collected last on purpose.
"""

import pytest
import torch

from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 6 << 20
PA_ERR_WORKSPACE = -4


def _both(b, case):
    d = P.dev(case)
    hkv, dim = case.num_kv_heads, case.head_dim
    ws = torch.zeros(b.pa_decode_balanced_workspace_bytes(case.batch, hkv, dim),
                     dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(d["q"])
    b.pa_decode_balanced(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                         d["context_lens"], case.scale, ws, ref)
    out = torch.full_like(d["q"], float("nan"))
    b.pa_decode_balanced_static(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], case.scale, out)
    torch.cuda.synchronize()
    return out, ref


def test_static_scratch_matches_workspace_entry_and_oracle_on_two_calls(cuda_lib):
    first = wl.make_case("static_a", 700, [3000, 5, 800, 0, 1234, 64, 4097, 17] * 6, 8, 2, 128,
                         16, append=False)
    second = wl.make_case("static_b", 701, [40, 2049, 1, 600] * 20, 16, 2, 128, 16,
                          append=False)
    for call, case in enumerate((first, second)):
        out, ref = _both(cuda_lib, case)
        got = P.to_f64(out)
        P.assert_close(got, P.to_f64(ref), f"call {call + 1} vs workspace entry")
        P.assert_close(got, P.oracle_out(case), f"call {call + 1} vs oracle")
    assert cuda_lib.pa_last_device_error() == 0


def test_static_scratch_refuses_shapes_beyond_its_size(cuda_lib):
    # 12000 sequences x 64 KV heads (G = 1) need more scratch than the array
    # holds; the call must return PA_ERR_WORKSPACE and leave `out` untouched.
    B, h, dim, bs = 12000, 64, 128, 16
    need = cuda_lib.pa_decode_balanced_workspace_bytes(B, h, dim)
    assert need > STATIC_SCRATCH_BYTES
    q = torch.zeros(B, h, dim, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, bs, h, dim, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    tables = torch.ones(B, 1, dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.full((B, h, dim), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.PagedKVError) as err:
        cuda_lib.pa_decode_balanced_static(q, kc, vc, tables, lens, 1.0 / dim ** 0.5, out)
    assert err.value.status == PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    # the refusal leaves the entry point usable
    small = wl.make_case("static_c", 702, [33, 1, 900], 8, 2, 128, 16, append=False)
    got, ref = _both(cuda_lib, small)
    P.assert_close(P.to_f64(got), P.oracle_out(small), "call after a refusal")
    assert cuda_lib.pa_last_device_error() == 0
