import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: long-running CPU case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The C-ABI library on a GPU; skips when no GPU is visible."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_45_gb300 import binding
    return binding


@pytest.fixture(params=["tcgen05", "columns"])
def multi_kernel(request, monkeypatch):
    """Short query chunks on the tcgen05 kernel (keys on M; the default where it
    applies: head_dim 128, block sizes >= 8, <= 32 columns per KV head, splits
    of 128 tokens) or on the column-warp kernel (PA_MULTI_KERNEL=columns)."""
    if request.param == "columns":
        monkeypatch.setenv("PA_MULTI_KERNEL", "columns")
    else:
        monkeypatch.delenv("PA_MULTI_KERNEL", raising=False)
    return request.param
