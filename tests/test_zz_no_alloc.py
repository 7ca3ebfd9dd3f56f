"""pa_decode_balanced_static: the decode entry point for callers that cannot
allocate device memory at the call site (an engine that has reserved its free
HBM for the KV block pool, a plug-in without an allocator). It uses the
library's built-in scratch array instead of a workspace.

Checked through the C ABI against pa_decode_balanced, the workspace entry
point, on two calls in a row with different batches, so the second call runs
on whatever the first left in the shared array. Tolerance: the parity bar of
the other tests (max abs <= 2e-2, per-row relative L2 <= 5e-3).

This file is collected last on purpose.
"""

import pytest
import torch

from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


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


def test_static_scratch_matches_workspace_entry_on_two_calls(cuda_lib):
    first = wl.make_case("static_a", 700, [3000, 5, 800, 0, 1234, 64, 4097, 17] * 6, 8, 2, 128,
                         16, append=False)
    second = wl.make_case("static_b", 701, [40, 2049, 1, 600] * 20, 16, 2, 128, 16,
                          append=False)
    for call, case in enumerate((first, second)):
        out, ref = _both(cuda_lib, case)
        P.assert_close(P.to_f64(out), P.to_f64(ref), f"call {call + 1}")
    assert cuda_lib.pa_last_device_error() == 0
