"""Failure detection without a GPU fault: a bounded wait that nothing
completes runs out, the kernel records it in the device error word and
returns, the host reads the status, and the context keeps working.
Bad tables are caught on the host (validating mode) in test_gpu_parity."""

import time

import pytest
import torch

from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_lost_wait_ends_in_a_status_not_a_hang(cuda_lib):
    b = cuda_lib
    assert b.pa_last_device_error() == 0
    t0 = time.perf_counter()
    b.pa_selftest_wait_timeout(20_000)          # 20 ms limit
    code = b.pa_last_device_error()             # synchronises, reads, clears
    elapsed = time.perf_counter() - t0
    assert code == 8, code
    assert elapsed < 5.0
    assert b.pa_last_device_error() == 0        # cleared by the read
    # the context is still usable: a decode right after matches the oracle
    case = wl.tiny_case(0)
    d = P.dev(case)
    b.pa_kv_append(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    out = b.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   case.scale, split_tokens=b.BALANCED)
    torch.cuda.synchronize()
    P.assert_close(P.to_f64(out), P.oracle_out(case), "after the self-test")


def test_selftest_rejects_bad_limits(cuda_lib):
    with pytest.raises(cuda_lib.PagedKVError):
        cuda_lib.pa_selftest_wait_timeout(0)
    with pytest.raises(cuda_lib.PagedKVError):
        cuda_lib.pa_selftest_wait_timeout(3_000_000)
