"""The bench's N > 1 host logic on CPU: two gloo ranks (127.0.0.1) combine
their step times and byte counts the way bench.py does on N GPUs, and the
reference arm leaves all work to rank 0."""

import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r: step time 1 + r seconds, 10 * (r + 1) bytes; e2e 2 + r s, 7 bytes
    stats = torch.tensor([1.0 + rank, 10.0 * (rank + 1), 2.0 + rank, 7.0, 0.0, 0.0],
                         dtype=torch.float64)
    out[rank] = bench.combine_ranks(stats)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_max_time_and_sum_bytes():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        total_s, alg_bytes, e2e_s, e2e_bytes = out[r]
        assert total_s == 2.0 and alg_bytes == 30.0      # slowest rank, all bytes
        assert e2e_s == 3.0 and e2e_bytes == 14.0


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
