"""The fused step (pa_append_decode) captured in a CUDA graph: after one eager
call has prepared the kernel, the entry point issues only its launch, so the
step can be recorded once and replayed; replays equal the eager step bit for
bit and follow new inputs written into the captured buffers."""

import numpy as np
import pytest
import torch

from paged_kv_cache_45_gb300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_fused_step_replays_from_a_cuda_graph(cuda_lib):
    b = cuda_lib
    case = wl.make_case("graph", 960, [100, 1000, 3000, 17, 0, 257] * 6, 8, 2, 128, 16)
    dv = P.dev(case)
    k0, v0 = dv["k_cache"].clone(), dv["v_cache"].clone()
    ws = torch.zeros(b.pa_decode_balanced_workspace_bytes(case.batch, 2, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(dv["q"])

    def step():
        b.pa_append_decode(dv["q"], dv["k_new"], dv["v_new"], dv["slot_mapping"], dv["k_cache"],
                           dv["v_cache"], dv["block_tables"], dv["context_lens"], case.scale, ws,
                           out)

    step()                                   # eager (also prepares the kernel)
    torch.cuda.synchronize()
    eager_out, eager_k = out.clone(), dv["k_cache"].clone()

    dv["k_cache"].copy_(k0)
    dv["v_cache"].copy_(v0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager_out.view(torch.int16))
    assert torch.equal(dv["k_cache"].view(torch.int16), eager_k.view(torch.int16))

    # new queries and new K/V rows into the captured buffers, replay again
    gen = torch.Generator().manual_seed(7)
    q2 = torch.randn(dv["q"].shape, generator=gen).to(torch.bfloat16)
    dv["q"].copy_(q2.cuda())
    g.replay()
    torch.cuda.synchronize()
    case.q = q2
    P.assert_close(P.to_f64(out), P.oracle_out(case), "graph replay with new q")
