#!/usr/bin/env python
"""Paged-KV GQA decode step on GB300: KV GB/s, % of HBM peak and steps/s.

Default workload: the 70B-shape continuous batch (B = 256 sequences, 64 query
heads on 8 KV heads, head_dim 128, bf16, block_size 16, context lengths
log-uniform in [128, 8192], each step every sequence finishes with p = 0.02
and a newcomer with a prompt log-uniform in [128, 2048] joins in its slot).
The 32-iteration schedule is drawn once and replayed cyclically (replays
re-write the same slots, so every step has the shape of its iteration).

A step is one pass of the hot path over the batch: the append of one new
token per sequence, then the decode over every sequence's paged context. By
default both run in one launch (pa_append_decode: the append fused into the
work-balanced decode); --step separate launches pa_kv_append and then
pa_decode_balanced, or pa_decode + pa_decode_splitk_reduce (--schedule split). Joiners' prompt rows (a prefill stand-in) are written with
pa_kv_append once before the warm-up and timed apart: they set block contents,
which the step's cost does not depend on. Inputs are resident in HBM; each
step streams ~1.7 GB of KV, far more than the 129 MB L2, so no L2 flush is
needed between steps.

  value   = algorithmic bytes (each attended token's K and V rows once, plus
            q in and out) / device time of the step (append + decode + reduce)
  e2e     = the same with the step's inputs copied from pinned host memory and
            the output copied back inside the timed region
  roofline: the decode kernel alone, timed with CUDA events around each of
            its launches on its stream (a separate instrumented pass).

--impl reference times the fp64 CPU oracle on the host cores instead (the
reference arm): each step is the oracle's append + decode of one sequence of
a sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-decode KV GB/s (% of GB300 HBM peak) and decode steps/s, 70B-shape batch"
FALLBACK_HBM_GBS = 6800.0
TIMED_SECONDS = 1.5   # wall time the repeated timed blocks aim for


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["cb70b", "8b", "long", "prefix", "spec", "prefill",
                                           "cow"],
                    default="cb70b",
                    help="spec: 4 query tokens per sequence (speculative verification, "
                         "pa_decode_multi); cow: the copy-on-write step of the prefix cache "
                         "(its own metric)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="fp8: the same workload on an e4m3 KV pool with per-head scales "
                         "(balanced schedule only)")
    ap.add_argument("--schedule", choices=["balanced", "split"], default="balanced",
                    help="balanced: pa_decode_balanced (one persistent launch); split: pa_decode "
                         "over fixed context splits + pa_decode_splitk_reduce")
    ap.add_argument("--step", choices=["fused", "separate"], default="fused",
                    help="fused: pa_append_decode (append + balanced decode in one launch); "
                         "separate: pa_kv_append, then the decode of --schedule")
    ap.add_argument("--multi-schedule", choices=["auto", "split", "balanced"], default="auto",
                    help="spec workload: pa_decode_multi over context splits (--split, default "
                         "1024) + reduce, or pa_decode_multi_balanced (one launch); auto: "
                         "balanced over bf16 caches, split over e4m3 pools")
    ap.add_argument("--split", type=int, default=-1,
                    help="split_tokens for --schedule split (-1: planned; 0: no split)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--repeats", type=int, default=0,
                    help="times the K-step block is timed (median reported); 0: enough blocks "
                         "for about 1.5 s of timed work, 3..200")
    ap.add_argument("--batch", type=int, default=256,
                    help="sequences of the continuous batch (256 is the workload; smaller "
                         "values are for profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=256)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the oracle's CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the pass that replays the timed steps from CUDA graphs")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# workloads as step lists (host side)
# ---------------------------------------------------------------------------

def describe(workload: str, batch: int = 256) -> str:
    return {
        "cb70b": "70B-shape continuous batching: B={batch}, 64 q heads / 8 KV heads, head_dim 128, "
                 "bf16, block_size 16, ctx log-uniform [128, 8192], p_finish 0.02, joiner "
                 "prompts log-uniform [128, 2048], 32-iteration schedule replayed",
        "8b": "8B-shape decode layer: B=64, 32 q heads / 8 KV heads, head_dim 128, bf16, "
              "block_size 16, ctx uniform [512, 4096] + 1 appended",
        "long": "long-context split-K: B=4 x 131072 tokens, 32 q heads / 8 KV heads, head_dim "
                "128, bf16, block_size 16, 1% of K rows x8, no append",
        "prefix": "radix prefix sharing: B=128, 2048-token prefix in the same 128 blocks, "
                  "private suffix uniform [64, 1024] + 1 appended, 8B heads",
        "prefill": "chunked prefill, 70B shape: 8 sequences each bringing a 2048-token chunk "
                   "after 6144 cached tokens (causal), 64 q heads / 8 KV heads, head_dim 128, "
                   "bf16, block_size 16; pa_kv_append of the chunk + pa_decode_multi "
                   "(tcgen05 kernel)",
        "spec": "speculative verification, 70B shape: B={batch} sequences, ctx log-uniform "
                "[128, 8192], 4 new query tokens each (causal), 64 q heads / 8 KV heads, "
                "head_dim 128, bf16, block_size 16; pa_kv_append of the 4 rows + "
                "pa_decode_multi",
        "cow": "copy-on-write after forking: {batch} sequences forked, the first append of "
               "each child copies its shared partial block (K and V, block_size 16, 8 KV heads, "
               "head_dim 128, bf16: 32 KiB each); 32 disjoint copy sets over a 1 GiB pool "
               "cycled",
    }[workload].replace("{batch}", str(batch))


def attended_pairs(q_start, context_lens) -> int:
    """(query row, key) pairs a causal multi-token step attends: sequence b's
    n_b rows sit at positions ctx_b - n_b .. ctx_b - 1 and row p sees keys
    0..p (none when p < 0): T(ctx_b) - T(max(ctx_b - n_b, 0)), T(x) = x(x+1)/2."""
    total = 0
    for b in range(len(context_lens)):
        n, c = int(q_start[b + 1]) - int(q_start[b]), int(context_lens[b])
        lo = max(c - n, 0)
        total += c * (c + 1) // 2 - lo * (lo + 1) // 2
    return total


class Steps:
    """Device-resident inputs of a workload's steps, cycled by index."""

    def __init__(self, workload: str, seed: int, device, batch: int = 256, kv_dtype="bf16"):
        import numpy as np
        import torch
        from paged_kv_cache_45_gb300 import workloads as wl
        self.workload = workload
        self.items = []
        self.fp8 = kv_dtype == "fp8"
        self.multi = workload in ("spec", "prefill")
        if self.multi:
            case = (wl.spec_verify_case(seed, batch=batch, q_len=4) if workload == "spec" else
                    prefill_case(seed))
            self.k_cache, self.v_cache = case.k_cache.to(device), case.v_cache.to(device)
            self.scale, self.hkv, self.hq, self.d = (case.scale, case.num_kv_heads,
                                                     case.num_q_heads, case.head_dim)
            self.max_context = int(case.block_tables.shape[1]) * case.block_size
            self.max_q_len = case.max_q_len
            self.block_size = case.block_size
            self.items.append(dict(fill=None, q=case.q, k_new=case.k_new, v_new=case.v_new,
                                   slots=case.slot_mapping, tables=case.block_tables,
                                   lens=case.context_lens, qstart=case.q_start))
            # attention FLOPs: 2 products x 2 FLOP x D per (row, attended key)
            attended = attended_pairs(case.q_start.numpy(), case.context_lens.numpy())
            self.items[-1]["flops"] = 4 * self.d * self.hq * attended
        elif workload == "cb70b":
            cb = wl.ContinuousBatching(seed=seed, batch=batch)
            self.cb = cb
            self.k_cache, self.v_cache = cb.initial_caches(device)
            self.scale, self.hkv, self.hq, self.d = cb.scale, cb.Hkv, cb.Hq, cb.D
            self.max_context = cb.max_blocks * cb.bs
            for it in range(cb.iterations):
                st = cb.step(it)
                self.items.append(dict(
                    fill=(st.fill_k.to(device), st.fill_v.to(device), st.fill_slots.to(device))
                    if st.fill_slots.numel() else None,
                    q=st.q, k_new=st.k_new, v_new=st.v_new, slots=st.slot_mapping,
                    tables=st.block_tables, lens=st.context_lens))
        else:
            case = {"8b": lambda: wl.llama8b_case(seed),
                    "long": lambda: wl.long_context_case(seed),
                    "prefix": lambda: wl.prefix_sharing_case(seed)}[workload]()
            self.k_cache, self.v_cache = case.k_cache.to(device), case.v_cache.to(device)
            self.scale, self.hkv, self.hq, self.d = (case.scale, case.num_kv_heads,
                                                     case.num_q_heads, case.head_dim)
            self.max_context = case.max_blocks * case.block_size
            self.items.append(dict(fill=None, q=case.q, k_new=case.k_new, v_new=case.v_new,
                                   slots=case.slot_mapping, tables=case.block_tables,
                                   lens=case.context_lens))
        for it in self.items:   # host copies (pinned) for e2e, device copies for the step
            it["host"] = {k: it[k].pin_memory() for k in ("q", "k_new", "v_new", "slots", "tables",
                                                           "lens", "qstart")
                          if it.get(k) is not None}
            it["dev"] = {k: v.to(device) for k, v in it["host"].items()}
            it["kv_bytes"] = (int(it["lens"].to(torch.int64).sum()) * 2 * self.hkv * self.d *
                              (1 if self.fp8 else 2))
            it["qo_bytes"] = 2 * it["q"].numel() * 2
        self.batch = int(self.items[0]["q"].shape[0])
        if self.fp8:   # e4m3 copy of the pool (per-KV-head scales), made on the device
            gen = np.random.Generator(np.random.PCG64(seed + 11_000))
            ks = (1.0 / 32.0 * (1.0 + 0.5 * gen.random(self.hkv))).astype(np.float32)
            vs = (1.0 / 32.0 * (1.0 + 0.5 * gen.random(self.hkv))).astype(np.float32)
            self.k_scale = torch.from_numpy(ks).to(device)
            self.v_scale = torch.from_numpy(vs).to(device)

            def codes(pool, sc):
                out = torch.empty(pool.shape, dtype=torch.uint8, device=device)
                for i in range(0, pool.shape[0], 4096):   # chunks: bounded temporaries
                    x = pool[i:i + 4096].float() / sc[:, None]
                    out[i:i + 4096] = x.to(torch.float8_e4m3fn).view(torch.uint8)
                return out
            self.k_cache = codes(self.k_cache, self.k_scale)
            self.v_cache = codes(self.v_cache, self.v_scale)
            torch.cuda.synchronize(device)

    def __len__(self):
        return len(self.items)


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int, period_ms: int = 20):
        self.proc = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    f"-lms={period_ms}", *sel]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), float(f[2]), f[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 0.3 * max(x[2] for x in rows)] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "power_w_max": max(r[2] for r in rows), "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {   # the files whose change invalidates a kernel's recorded DRAM traffic
    "balanced_decode_kernel": ("pa_decode_balanced.cu", "pa_balance.cuh", "pa_tile.cuh",
                               "pa_device.cuh", "pa_api.cu"),
    "balanced_decode_kernel[e4m3]": ("pa_decode_balanced.cu", "pa_balance.cuh", "pa_tile.cuh",
                                     "pa_device.cuh", "pa_api.cu"),
    "paged_decode_kernel": ("pa_decode.cu", "pa_tile.cuh", "pa_device.cuh", "pa_api.cu"),
    "multi_decode_kernel": ("pa_decode_multi.cu", "pa_tile.cuh", "pa_device.cuh", "pa_api.cu"),
    "multi_decode_kernel[e4m3]": ("pa_decode_multi.cu", "pa_tile.cuh", "pa_device.cuh",
                                  "pa_api.cu"),
    "balanced_multi_kernel": ("pa_decode_multi.cu", "pa_balance.cuh", "pa_tile.cuh",
                              "pa_device.cuh", "pa_api.cu"),
    "rowblock_decode_kernel": ("pa_decode_multi.cu", "pa_tile.cuh", "pa_device.cuh",
                               "pa_api.cu"),
    "prefill_tc_kernel": ("pa_prefill_tc.cu", "pa_tc_common.cuh", "pa_umma.cuh",
                          "pa_device.cuh"),
    "prefill_tc_kernel[e4m3]": ("pa_prefill_tc.cu", "pa_tc_common.cuh", "pa_umma.cuh",
                                "pa_device.cuh"),
    "verify_tc_kernel": ("pa_verify_tc.cu", "pa_tc_common.cuh", "pa_umma.cuh", "pa_device.cuh",
                         "pa_balance.cuh"),
    "verify_tc_kernel[balanced]": ("pa_verify_tc.cu", "pa_tc_common.cuh", "pa_umma.cuh",
                                   "pa_device.cuh", "pa_balance.cuh"),
}


def multi_kernel_name(steps, ws) -> str:
    """The kernel pa_decode_multi(_fp8) runs for a short-chunk step: the
    tcgen05 keys-on-M kernel for bf16 caches (head_dim 128, block sizes >= 8,
    <= 32 (token, head) columns per KV head, splits of 128 tokens), else the
    column-warp kernel."""
    if steps.fp8:
        return "multi_decode_kernel[e4m3]"
    tc = (steps.d == 128 and steps.block_size >= 8
          and steps.max_q_len * (steps.hq // steps.hkv) <= 32
          and ws.split_tokens % 128 == 0
          and os.environ.get("PA_MULTI_KERNEL") != "columns")
    if ws.multi_balanced:
        return "verify_tc_kernel[balanced]" if tc and steps.batch <= 8192 else \
            "balanced_multi_kernel"
    return "verify_tc_kernel" if tc else "multi_decode_kernel"


class MultiWorkspace:
    """Output and split-mode buffers of pa_decode_multi (rows, not sequences)."""

    def __init__(self, b, steps, split, device):
        import torch
        R = int(steps.items[0]["q"].shape[0])
        self.balanced = False
        self.multi_balanced = split < 0
        split = max(split, 0)
        self.scratch = torch.zeros(b.pa_decode_multi_balanced_workspace_bytes(
            steps.batch, steps.hkv, steps.d), dtype=torch.uint8, device=device) \
            if self.multi_balanced else None
        self.split_tokens = split
        self.max_splits = b.pa_decode_num_splits(steps.max_context, split) if split else 0
        self.out = torch.empty((R, steps.hq, steps.d), dtype=torch.bfloat16, device=device)
        S = max(self.max_splits, 1)
        self.part_out = torch.empty((R, steps.hq, S, steps.d), dtype=torch.float32,
                                    device=device) if split else None
        self.part_lse = torch.empty((R, steps.hq, S), dtype=torch.float32,
                                    device=device) if split else None
        self.row_lens = torch.empty(R, dtype=torch.int32, device=device) if split else None


def code_of(text: str) -> str:
    """C/CUDA source with comments and blank lines removed and each line's
    whitespace collapsed: what the compiler sees, so that editing a comment
    keeps a capture valid."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(re.sub(r"\s+", " ", line.strip()) for line in text.splitlines()
                     if line.strip())


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_cache_45_gb300", "csrc", name)) as fh:
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def library_source_hash() -> str:
    """sha256 (16 hex digits) of the library's whole source (csrc and the
    public header, comments and blank lines removed), so that a recorded bench
    line can be matched with the code that produced it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_45_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)
                   if f.endswith((".cu", ".cuh", ".h", ".cpp")))
    files.append(os.path.join(ROOT, "include", "pagedkv.h"))
    for path in files:
        with open(path) as fh:
            h.update(os.path.basename(path).encode())
            h.update(code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(kernel: str, kv_tokens_per_launch: float):
    """DRAM read+write bytes of one decode launch, scaled by KV tokens from the
    ncu capture recorded in profiles/dram_traffic.txt, if that capture was
    taken on the current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as fh:
            for line in fh:
                f = line.split()
                if len(f) >= 3 and not line.startswith("#") and f[0] == kernel:
                    if f[1] != kernel_source_hash(kernel):
                        return None
                    return float(f[2]) * kv_tokens_per_launch
    except OSError:
        pass
    return None


def combine_ranks(stats):
    """Whole-job figures from per-rank [time_s, bytes, e2e_time_s, e2e_bytes, ...]:
    the slowest rank's times (max) and every rank's bytes (sum). Collective
    over the default process group (NCCL on GPUs; gloo works on CPU)."""
    import torch.distributed as dist
    mx, sm = stats.clone(), stats.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[1]), float(mx[2]), float(sm[3])


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    from paged_kv_cache_45_gb300 import binding as b

    # the oracle's CPU baseline runs first, in a fresh process with one BLAS thread
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_subprocess(args)

    steps = Steps(args.workload, args.seed + rank, device, args.batch, args.kv_dtype)
    if steps.fp8 and not steps.multi and args.schedule != "balanced":
        raise SystemExit("--kv-dtype fp8 runs the balanced schedule only")
    if args.multi_schedule == "auto":
        args.multi_schedule = "split" if steps.fp8 or args.split >= 0 else "balanced"
    if steps.fp8 and steps.multi and args.multi_schedule == "balanced":
        raise SystemExit("--kv-dtype fp8 with several query tokens runs the split schedule "
                         "(--workload spec, --workload prefill) only")
    sms = b.num_sms(local)
    if steps.multi:   # -1: the balanced schedule (pa_decode_multi_balanced)
        split = -1 if args.multi_schedule == "balanced" else (args.split if args.split >= 0
                                                              else 1024)
        if args.workload == "prefill":
            split = 0     # long chunks run unsplit (the tcgen05 kernel)
    elif args.schedule == "balanced":
        split = b.BALANCED
    elif args.split >= 0:
        split = args.split
    elif args.workload == "long":
        split = 4096
    else:
        split = max(b.plan_split(it["lens"].numpy(), steps.hkv, sms) for it in steps.items)
    if steps.multi:
        ws = MultiWorkspace(b, steps, split, device)
    else:
        ws = b.DecodeWorkspace(steps.batch, steps.hq, steps.d, split, steps.max_context, device,
                               num_kv_heads=steps.hkv)
    stream = torch.cuda.current_stream(device)

    def fill(it):
        if it["fill"] is not None:
            fk, fv, fs = it["fill"]
            if steps.fp8:
                b.pa_kv_append_fp8(fk, fv, fs, steps.k_cache, steps.v_cache, steps.k_scale,
                                   steps.v_scale)
            else:
                b.pa_kv_append(fk, fv, fs, steps.k_cache, steps.v_cache)

    fused = args.step == "fused" and ws.balanced and steps.items[0]["dev"].get("k_new") is not None

    def step(dv, ev=None):
        if steps.multi:
            if ev is not None:
                ev[0].record(stream)
            if steps.fp8:
                b.pa_kv_append_fp8(dv["k_new"], dv["v_new"], dv["slots"], steps.k_cache,
                                   steps.v_cache, steps.k_scale, steps.v_scale)
            else:
                b.pa_kv_append(dv["k_new"], dv["v_new"], dv["slots"], steps.k_cache,
                               steps.v_cache)
            if ev is not None:
                ev[1].record(stream)
            if steps.fp8:
                b.pa_decode_multi_fp8(dv["q"], steps.k_cache, steps.v_cache, steps.k_scale,
                                      steps.v_scale, dv["tables"], dv["lens"], dv["qstart"],
                                      steps.max_q_len, steps.scale, ws.out, ws.split_tokens,
                                      ws.max_splits, ws.part_out, ws.part_lse, ws.row_lens)
            elif ws.multi_balanced:
                b.pa_decode_multi_balanced(dv["q"], steps.k_cache, steps.v_cache, dv["tables"],
                                           dv["lens"], dv["qstart"], steps.max_q_len,
                                           steps.scale, ws.scratch, ws.out)
            else:
                b.pa_decode_multi(dv["q"], steps.k_cache, steps.v_cache, dv["tables"],
                                  dv["lens"], dv["qstart"], steps.max_q_len, steps.scale,
                                  ws.out, ws.split_tokens, ws.max_splits, ws.part_out,
                                  ws.part_lse, ws.row_lens)
            if ev is not None:
                ev[2].record(stream)
            if ws.split_tokens:
                b.pa_decode_splitk_reduce(ws.part_out, ws.part_lse, ws.row_lens, ws.split_tokens,
                                          ws.out)
            if ev is not None:
                ev[3].record(stream)
            return
        if fused:
            if ev is not None:
                ev[0].record(stream)
                ev[1].record(stream)
            if steps.fp8:
                b.pa_append_decode_fp8(dv["q"], dv["k_new"], dv["v_new"], dv["slots"],
                                       steps.k_cache, steps.v_cache, steps.k_scale,
                                       steps.v_scale, dv["tables"], dv["lens"], steps.scale,
                                       ws.scratch, ws.out)
            else:
                b.pa_append_decode(dv["q"], dv["k_new"], dv["v_new"], dv["slots"],
                                   steps.k_cache, steps.v_cache, dv["tables"], dv["lens"],
                                   steps.scale, ws.scratch, ws.out)
            if ev is not None:
                ev[2].record(stream)
                ev[3].record(stream)
            return
        if ev is not None:
            ev[0].record(stream)
        if dv.get("k_new") is not None:
            if steps.fp8:
                b.pa_kv_append_fp8(dv["k_new"], dv["v_new"], dv["slots"], steps.k_cache,
                                   steps.v_cache, steps.k_scale, steps.v_scale)
            else:
                b.pa_kv_append(dv["k_new"], dv["v_new"], dv["slots"], steps.k_cache,
                               steps.v_cache)
        if ev is not None:
            ev[1].record(stream)
        if ws.balanced:
            if steps.fp8:
                b.pa_decode_balanced_fp8(dv["q"], steps.k_cache, steps.v_cache, steps.k_scale,
                                         steps.v_scale, dv["tables"], dv["lens"], steps.scale,
                                         ws.scratch, ws.out)
            else:
                b.pa_decode_balanced(dv["q"], steps.k_cache, steps.v_cache, dv["tables"],
                                     dv["lens"], steps.scale, ws.scratch, ws.out)
        else:
            b.pa_decode(dv["q"], steps.k_cache, steps.v_cache, dv["tables"], dv["lens"],
                        steps.scale, ws.out, ws.split_tokens, ws.max_splits, ws.part_out,
                        ws.part_lse)
        if ev is not None:
            ev[2].record(stream)
        if ws.split_tokens:
            b.pa_decode_splitk_reduce(ws.part_out, ws.part_lse, dv["lens"], ws.split_tokens, ws.out)
        if ev is not None:
            ev[3].record(stream)

    n = len(steps)
    # Joiners' prompt rows (the prefill stand-in) are written once, before the
    # warm-up: they only set block contents, which the decode step's cost does
    # not depend on; their time is reported apart from the step.
    fill_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    fill_ev[0].record(stream)
    n_fills = 0
    for it in steps.items:
        if it["fill"] is not None:
            fill(it)
            n_fills += 1
    fill_ev[1].record(stream)
    for w in range(args.warmup):
        step(steps.items[w % n]["dev"])
    torch.cuda.synchronize()
    fill_ms = fill_ev[0].elapsed_time(fill_ev[1])

    # ------------------------------------------------ the timed region: K steps
    K = args.steps
    idx = [(args.warmup + k) % n for k in range(K)]
    per_step_launches = 1 if fused else \
        (1 if steps.items[0]["dev"].get("k_new") is not None else 0) + 1 + (1 if ws.split_tokens else 0)
    # The block of K steps is timed several times back to back (each bracketed
    # by a barrier and a synchronize) and the median block is reported, so
    # that even a short K spans enough wall time for the clock sampler: the
    # repeats after the first fill about TIMED_SECONDS.
    t_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.__enter__()
    block_s, repeats = [], args.repeats
    t_wall0 = time.perf_counter()
    while len(block_s) < max(repeats, 1):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_ev[0].record(stream)
        for k in range(K):
            step(steps.items[idx[k]]["dev"])
        t_ev[1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        block_s.append(t_ev[0].elapsed_time(t_ev[1]) / 1e3)
        if len(block_s) == 1 and repeats <= 0:   # automatic: from the first block
            want = min(200, max(3, math.ceil(TIMED_SECONDS / max(block_s[0], 1e-6))))
            if world > 1:   # every rank runs the same number of blocks
                w_t = torch.tensor([want], dtype=torch.int64, device=device)
                dist.all_reduce(w_t, op=dist.ReduceOp.MAX)
                want = int(w_t.item())
            repeats = want
    t_wall = time.perf_counter() - t_wall0
    if sampler:
        sampler.__exit__(None, None, None)
    launches = K * per_step_launches
    total_s = statistics.median(block_s)
    alg_bytes = sum(steps.items[i]["kv_bytes"] + steps.items[i]["qo_bytes"] for i in idx)

    # ------------------ the same K steps replayed from CUDA graphs (one graph
    # per distinct step input, captured after the warm-up: a warmed entry point
    # issues only its launches)
    graph_s = None
    if not args.no_graph:
        graphs = []
        for it in steps.items:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(it["dev"])
            graphs.append(g)
        for w in range(3):
            graphs[w % n].replay()
        g_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        g_ev[0].record(stream)
        for k in range(K):
            graphs[idx[k]].replay()
        g_ev[1].record(stream)
        torch.cuda.synchronize()
        graph_s = g_ev[0].elapsed_time(g_ev[1]) / 1e3
        del graphs

    # ---------- an instrumented pass: events around every launch of the step
    # (the per-kernel breakdown and the decode kernel's own duration; an event
    # pair costs ~2 us of device time, so these steps are not the headline)
    KI = min(K, 512)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KI)]
    for k in range(KI):
        step(steps.items[idx[k]]["dev"], evs[k])
    torch.cuda.synchronize()
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    app_ms = [e[0].elapsed_time(e[1]) for e in evs]
    red_ms = [e[2].elapsed_time(e[3]) for e in evs]
    dec_bytes = sum(steps.items[idx[k]]["kv_bytes"] + steps.items[idx[k]]["qo_bytes"]
                    for k in range(KI))
    kv_tokens = sum(int(steps.items[idx[k]]["lens"].sum()) for k in range(KI))
    dec_s = sum(dec_ms) / 1e3

    # ------------------------------------------------------------ end to end
    # Each step's inputs start in pinned host memory, packed in one buffer (one
    # H2D copy), and its output ends in pinned host memory. Double-buffered on
    # three streams -- H2D of step k+1 and D2H of step k-1 overlap step k's
    # kernels, as a serving loop would run them; the timed region spans the
    # first H2D to the last D2H.
    E = min(args.e2e_steps, K)
    keys = [k for k in ("q", "k_new", "v_new", "slots", "tables", "lens", "qstart")
            if k in steps.items[0]["host"]]

    def layout(host):
        offs, off = {}, 0
        for key in keys:
            offs[key] = off
            off += (host[key].numel() * host[key].element_size() + 255) // 256 * 256
        return offs, off

    packed = []
    for it in steps.items:
        offs, total = layout(it["host"])
        buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
        for key in keys:
            t = it["host"][key]
            nbytes = t.numel() * t.element_size()
            buf[offs[key]:offs[key] + nbytes].copy_(t.contiguous().view(-1).view(torch.uint8))
        packed.append((buf, offs))
    cap_bytes = max(b_.numel() for b_, _ in packed)
    dev_in = [torch.empty(cap_bytes, dtype=torch.uint8, device=device) for _ in range(2)]

    def views(dbuf, offs, like):
        v = {}
        for key in keys:
            t = like[key]
            nbytes = t.numel() * t.element_size()
            v[key] = dbuf[offs[key]:offs[key] + nbytes].view(t.dtype).view(t.shape)
        return v

    out_ring = [torch.empty_like(ws.out) for _ in range(2)]
    out_host = [torch.empty(ws.out.shape, dtype=ws.out.dtype, pin_memory=True) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {name: [torch.cuda.Event() for _ in range(2)]
          for name in ("h2d", "free", "out", "d2h")}
    bi = packed[0][0].numel()
    bo = out_host[0].numel() * out_host[0].element_size()
    e2e_bytes = sum(steps.items[k % n]["kv_bytes"] + steps.items[k % n]["qo_bytes"]
                    for k in range(E))
    e2e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    e2e_ev[0].record(stream)
    h2d_s.wait_event(e2e_ev[0])
    for k in range(E):
        s_ = k % 2
        buf, offs = packed[k % n]
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(ev["free"][s_])           # step k-2 is done with dev_in[s_]
            dev_in[s_][:buf.numel()].copy_(buf, non_blocking=True)
            ev["h2d"][s_].record(h2d_s)
        stream.wait_event(ev["h2d"][s_])
        step(views(dev_in[s_], offs, steps.items[k % n]["host"]))
        stream.wait_event(ev["d2h"][s_])                 # out_ring[s_] was read back
        out_ring[s_].copy_(ws.out, non_blocking=True)
        ev["free"][s_].record(stream)
        ev["out"][s_].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev["out"][s_])
            out_host[s_].copy_(out_ring[s_], non_blocking=True)
            ev["d2h"][s_].record(d2h_s)
    stream.wait_event(ev["d2h"][(E - 1) % 2])
    e2e_ev[1].record(stream)
    torch.cuda.synchronize()
    e2e_s = e2e_ev[0].elapsed_time(e2e_ev[1]) / 1e3

    # ------------------------------------------------------------ across ranks
    graph_line = None
    if graph_s is not None:
        graph_line = {"ms_per_step": round(graph_s / K * 1e3, 5),
                      "value": round(alg_bytes / world / graph_s / 1e9, 2), "unit": "GB/s",
                      "graphs": n, "note": "the same K steps replayed from CUDA graphs "
                                           "(one per distinct step input), rank 0"}
    stats = torch.tensor([total_s, alg_bytes, e2e_s, e2e_bytes, dec_s, dec_bytes],
                         dtype=torch.float64, device=device)
    if world > 1:
        total_s, alg_bytes, e2e_s, e2e_bytes = combine_ranks(stats)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_hbm_peak()
    gbs = alg_bytes / total_s / 1e9
    dec_gbs_rank0 = dec_bytes / dec_s / 1e9
    kv_tokens_per_launch = kv_tokens / KI
    kernel = ("balanced_decode_kernel" + ("[e4m3]" if steps.fp8 else "")) if ws.balanced \
        else (multi_kernel_name(steps, ws)
              if steps.multi else "paged_decode_kernel")
    if args.workload == "prefill":
        kernel = ("rowblock_decode_kernel" if os.environ.get("PA_PREFILL_KERNEL") == "rowblock"
                  and not steps.fp8 else
                  "prefill_tc_kernel" + ("[e4m3]" if steps.fp8 else ""))
    traffic = traffic_per_launch(kernel, kv_tokens_per_launch)
    clocks = sampler.summary() if sampler else None
    prefill = args.workload == "prefill"
    if prefill:   # compute-bound: TFLOP/s against the measured bf16 tensor peak
        flops = steps.items[0]["flops"]
        tflops = flops * K / total_s / 1e12
        kern_tflops = flops * KI / dec_s / 1e12
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
                tpeak, tkind = float(json.load(fh)["bf16_tflops"]), "measured"
        except Exception:
            tpeak, tkind = 1900.0, "fallback"
    line = {
        "metric": PREFILL_METRIC if prefill else METRIC,
        "value": round(tflops, 2) if prefill else round(gbs, 2),
        "unit": "TFLOP/s" if prefill else "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_s / K * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 KV, bf16 q/out" if steps.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/K/V; seeded lengths and block placement)",
        "config": {"workload": describe(args.workload, args.batch) +
                   (" (e4m3 KV pool, per-KV-head scales)" if steps.fp8 else ""),
                   "schedule": ("row blocks (64 (token, head) rows x KV head x sequence per "
                                "block, unsplit, mma.sync)"
                                if os.environ.get("PA_PREFILL_KERNEL") == "rowblock" else
                                "tcgen05 blocks (256 (token, head) rows x KV head x sequence, "
                                "unsplit)") if args.workload == "prefill" else
                   "balanced" if ws.balanced else
                   ((("multi, balanced persistent (pa_decode_multi_balanced) on the tcgen05 "
                      "keys-on-M kernel: equal ranges of 128-key tiles, cut units merged in "
                      "the kernel"
                      if multi_kernel_name(steps, ws) == "verify_tc_kernel[balanced]" else
                      "multi, balanced persistent (pa_decode_multi_balanced)")
                     if ws.multi_balanced else
                     (f"multi, tcgen05 keys-on-M kernel (persistent, one block per SM, units "
                      f"of (sequence, split, KV head); split_tokens={ws.split_tokens})"
                      if multi_kernel_name(steps, ws) == "verify_tc_kernel" else
                      f"multi (one block per KV head, split, sequence; split_tokens="
                      f"{ws.split_tokens})")) if steps.multi else
                    f"split (pa_decode split_tokens={ws.split_tokens} + pa_decode_splitk_reduce)"),
                   "step": "fused: pa_append_decode, one launch" if fused else
                   "separate: pa_kv_append + decode launches",
                   "split_tokens": ws.split_tokens, "max_splits": ws.max_splits,
                   "batch": steps.batch,
                   "l2": "no flush: each step reads ~2 GB of KV, inputs far larger than the 129 MB L2"
                   if args.workload == "cb70b" else "inputs larger than L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_peak": round(100 * gbs / peak, 2),
        "steps_per_s": round(K / total_s, 1),
        "kv_bytes_per_step": int(alg_bytes / K / world),
        "pct_of_datasheet_8tbs": round(100 * gbs / 8000.0, 2),
        "ms_breakdown": {"append": None if fused else round(statistics.mean(app_ms), 5),
                         "decode": round(statistics.mean(dec_ms), 5),
                         "reduce_or_event_gap": round(statistics.mean(red_ms), 5),
                         "steps": KI, "note": "instrumented pass, an event pair around each "
                                             "launch"},
        "fill_ms_before_warmup": round(fill_ms, 4), "fills": n_fills,
        "roofline": {"bound": "hbm", "kernel": kernel,
                     "achieved": round(dec_gbs_rank0, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(dec_gbs_rank0 / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "traffic": None if traffic is None else int(traffic),
                     "algorithmic_bytes_per_launch": int(dec_bytes / KI),
                     "measured": f"CUDA events around each decode launch, {KI} steps"},
        "e2e": {"value": round(e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo), "steps": E,
                "note": "inputs packed in one pinned buffer (one H2D copy a step), output read "
                        "back to pinned memory; double-buffered on three streams so the copies "
                        "of neighbouring steps overlap each step's kernels"},
        "gpu_launches": launches,
        "source_sha16": library_source_hash(),
        "timed_blocks": {"blocks": len(block_s), "ms_per_step_min": round(min(block_s) / K * 1e3, 5),
                         "ms_per_step_median": round(total_s / K * 1e3, 5),
                         "ms_per_step_max": round(max(block_s) / K * 1e3, 5),
                         "note": "the K-step block timed back to back this many times; value and "
                                 "ms_per_step are the median block's; gpu_launches counts one "
                                 "block"},
        "wall_s_timed_region": round(t_wall, 4),
        "timing": "CUDA events bracketing each block of K steps on the launching stream, "
                  "barrier + synchronize on both sides; the median block is reported",
    }
    if prefill:
        line["roofline"] = {
            "bound": "tensor", "kernel": kernel, "achieved": round(kern_tflops, 2),
            "peak": tpeak, "unit": "TFLOP/s", "frac": round(kern_tflops / tpeak, 4),
            "peak_kind": f"{tkind} bf16_tflops (cuBLAS burst)" +
                         ("; the e4m3 pool's MMAs run f16, whose dense rate is bf16's"
                          if steps.fp8 else ""),
            "traffic": None if traffic is None else int(traffic),
            "algorithmic_flops_per_launch": int(flops),
            "measured": f"CUDA events around each decode launch, {KI} steps"}
        line["kv_gbs"] = round(gbs, 2)
        line["e2e"]["value"] = round(flops * E / e2e_s / 1e12, 2)
        line["e2e"]["unit"] = "TFLOP/s"
        line["config"]["l2"] = ("inputs larger than L2: 134 MB of e4m3 K/V read every step"
                                if steps.fp8 else
                                "inputs larger than L2: 268 MB of K/V read every step")
        line.pop("pct_of_hbm_peak", None)
        line.pop("pct_of_datasheet_8tbs", None)
    if graph_line is not None:
        if prefill:
            graph_line["value"] = round(steps.items[0]["flops"] * K / graph_s / 1e12, 2)
            graph_line["unit"] = "TFLOP/s"
        line["graph"] = graph_line
    if clocks is not None:
        line["clocks"] = clocks
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if getattr(steps, "cb", None) is not None and rank == 0:
        host_ms = host_bookkeeping_ms(steps.cb)
        e2e_ms = e2e_s / E * 1e3
        line["host_bookkeeping"] = {
            "ms_per_step": round(host_ms, 4), "steps": steps.cb.iterations,
            "what": "the step's host side on the native prefix cache (pa_prefix_*): finished "
                    "sequences discarded, joiners admitted with their prompt slots, one decode "
                    "slot per sequence, block tables and lengths (median over the schedule)",
            "wall_steps_per_s_serial": round(1e3 / (host_ms + e2e_ms), 1),
            "note": "serial bound: the host work, then the e2e step (H2D of the step's inputs "
                    "with its tables, the kernels, D2H of the output); a serving loop overlaps "
                    "the two"}
        p_ms, p_ev = host_bookkeeping_ms(steps.cb, pressure=True)
        line["host_bookkeeping_pressure"] = {
            "ms_per_step": round(p_ms, 4), "evicted_blocks_per_step": round(p_ev, 1),
            "what": "the same steps with the pool full of cached prefixes: joiners share 8 "
                    "system prompts of 512 tokens, finished sequences are released into the "
                    "cache, and fresh blocks come mostly from LRU eviction",
            "wall_steps_per_s_serial": round(1e3 / (p_ms + e2e_ms), 1)}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def host_bookkeeping_ms(cb, pressure: bool = False):
    """Median host time of one continuous-batching step's scheduler work on
    the native prefix cache, replaying the schedule's finishes and joins:
    discard the finished sequences, admit each joiner's prompt (a token
    stream no other sequence shares, so nothing is matched) and take its
    slots, one decode slot per running sequence, then the block tables and
    context lengths. The lengths must equal the schedule's.

    pressure=True: the serving case where the prefix cache has filled the
    pool. Before the first step every free block is taken by cached, unused
    prefixes; joiners' prompts begin with one of 8 shared 512-token system
    prompts; finished sequences are released with their tokens (their full
    blocks stay cached; their partial last blocks go back to the free
    list). The fresh blocks a step takes then come mostly from evicting the
    least recently used unreferenced prefixes ([PYS] "The radix prefix
    cache"). Returns (median ms, blocks evicted per step on average)."""
    import numpy as np
    from paged_kv_cache_45_gb300 import binding as b
    pc = b.PrefixCache(cb.num_blocks, cb.bs)
    uid = [0]
    sys_len = 512
    systems = [(1 << 30) + (k << 13) + np.arange(sys_len, dtype=np.int32) for k in range(8)]

    def private(u, p0, p1):
        return (u << 13) + np.arange(p0, p1, dtype=np.int32)   # positions < 8192 = 2^13

    def prompt(n, shared):
        uid[0] += 1
        if not shared:
            return uid[0], -1, private(uid[0], 0, n)
        k = uid[0] % len(systems)
        s = min(sys_len, n - 1)
        return uid[0], k, np.concatenate([systems[k][:s], private(uid[0], s, n)])

    def tokens_of(u, k, n):     # a sequence's tokens after n positions
        if k < 0:
            return private(u, 0, n)
        s = min(sys_len, n)
        return np.concatenate([systems[k][:s], private(u, s, n)])

    try:
        ids = np.zeros(cb.B, dtype=np.int64)
        who = [None] * cb.B        # (uid, system prompt or -1) of each slot's sequence
        for i in range(cb.B):      # the running batch before the first iteration (untimed)
            n = int(cb.initial_lens[i])
            u, k, toks = prompt(n, False)
            sid, cached = pc.admit(toks)
            pc.write_slots(sid, cached, n)
            ids[i] = sid
            who[i] = (u, k)
        if pressure:               # fill the pool with cached, unreferenced prefixes
            while pc.stats()[0] > 0:
                n = min(2048, pc.stats()[0] * cb.bs)
                _, _, toks = prompt(n, False)
                sid, cached = pc.admit(toks)
                pc.write_slots(sid, cached, n)
                pc.release(sid, toks)
        times, evicted = [], 0
        for it in range(cb.iterations):
            sch = cb.schedule[it]
            fin = sch["finished"]
            prev = cb.initial_lens if it == 0 else cb.schedule[it - 1]["lens"].numpy()
            done = [tokens_of(*who[i], int(prev[i])) for i in fin] if pressure else []
            joins = [(seq, plen) + prompt(plen, pressure) for seq, plen in sch["joins"]]
            cached0 = pc.stats()[1]
            t0 = time.perf_counter()
            if fin:
                if pressure:
                    for i, toks in zip(fin, done):
                        pc.release(int(ids[i]), toks)
                else:
                    pc.discard(ids[fin])
                for seq, plen, u, k, toks in joins:
                    sid, cached = pc.admit(toks)
                    pc.write_slots(sid, cached, plen)
                    ids[seq] = sid
                    who[seq] = (u, k)
            pc.append_tokens(ids)
            _, lens = pc.tables(ids, cb.max_blocks)
            times.append(time.perf_counter() - t0)
            if not np.array_equal(lens, sch["lens"].numpy()):
                raise RuntimeError(f"prefix cache lengths differ from the schedule at step {it}")
            if pressure:
                # blocks cached by this step's releases, minus those still cached
                added = sum(len(t) // cb.bs for t in done)
                evicted += max(cached0 + added - pc.stats()[1], 0)
        ms = statistics.median(times) * 1e3
        return (ms, evicted / cb.iterations) if pressure else ms
    finally:
        pc.close()


# ---------------------------------------------------------------------------
# the oracle on the host cores: CPU baseline and the reference arm
# ---------------------------------------------------------------------------

def prefill_case(seed: int, n_seqs: int = 8):
    """The chunked-prefill step: n_seqs sequences, 6144 cached + 2048 new tokens."""
    from paged_kv_cache_45_gb300 import workloads as wl
    return wl.make_multi_case("prefill", seed, [6144] * n_seqs, [2048] * n_seqs, 64, 8, 128, 16)


def prefill_cpu_baseline(seed: int, budget_s: float):
    """The oracle's decode_multi on the host over a bounded sample of the
    prefill step: the chunk's rows of one sequence, taken in order, each row
    at its own causal context (row i of the chunk sees 6144 + i + 1 keys)."""
    import numpy as np
    import oracle
    from oracle import paged_attention as pa
    from paged_kv_cache_45_gb300 import workloads as wl
    case = prefill_case(seed, n_seqs=1)
    kc, vc = pa.kv_append(wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.k_new),
                          wl.bits(case.v_new), case.slot_mapping.numpy())
    q, bt = wl.bits(case.q), case.block_tables.numpy()
    n, ctx = int(case.q_start[1]), int(case.context_lens[0])
    flops, secs, rows = 0, 0.0, 0
    while rows < n and (secs < budget_s or rows < 2):
        pos = ctx - n + rows
        t0 = time.perf_counter()
        oracle.decode_multi(q[rows:rows + 1], kc, vc, bt, np.array([pos + 1]),
                            np.array([0, 1]), case.scale)
        secs += time.perf_counter() - t0
        flops += 4 * case.head_dim * case.num_q_heads * (pos + 1)
        rows += 1
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle",
            "sample": f"the first {rows} rows of one sequence's 2048-token chunk (each at its "
                      f"causal context, 6145.. keys, 64 heads), fp64 oracle decode_multi, "
                      f"{blas_threads()} BLAS thread(s), {secs:.1f} s"}


def oracle_sample_case(seed: int, n_seqs: int = 48):
    """A bounded sample of the 70B-shape batch: n_seqs sequences with lengths
    drawn from the same log-uniform [128, 8192] law, one appended token."""
    import numpy as np
    from paged_kv_cache_45_gb300 import workloads as wl
    rng = np.random.Generator(np.random.PCG64(seed + 3_000))
    lens = wl.loguniform(rng, 128, 8192, n_seqs)
    return wl.make_case("cb70b_sample", seed, lens, 64, 8, 128, 16)


def oracle_steps(case, budget_s: float, max_steps: int | None = None):
    """Time the oracle's append + decode of one sequence per step."""
    from oracle import paged_attention as pa
    from paged_kv_cache_45_gb300 import workloads as wl
    q, kc, vc = wl.bits(case.q), wl.bits(case.k_cache), wl.bits(case.v_cache)
    kn, vn = wl.bits(case.k_new), wl.bits(case.v_new)
    bt, cl, slots = case.block_tables.numpy(), case.context_lens.numpy(), case.slot_mapping.numpy()
    per_tok = 2 * case.num_kv_heads * case.head_dim * 2
    times, nbytes = [], []
    t_start = time.perf_counter()
    i = 0
    while True:
        b = i % case.batch
        t0 = time.perf_counter()
        pa.kv_append_inplace(kc, vc, kn[b:b + 1], vn[b:b + 1], slots[b:b + 1])
        pa.decode(q, kc, vc, bt, cl, case.scale, seqs=[b])
        times.append(time.perf_counter() - t0)
        nbytes.append(int(cl[b]) * per_tok + 2 * case.num_q_heads * case.head_dim * 2)
        i += 1
        if max_steps is not None and i >= max_steps:
            break
        if max_steps is None and time.perf_counter() - t_start > budget_s:
            break
    return times, nbytes


def cpu_baseline_child(seed: int, budget_s: float) -> None:
    case = oracle_sample_case(seed)
    times, nbytes = oracle_steps(case, budget_s)
    print(json.dumps({"value": round(sum(nbytes) / sum(times) / 1e9, 4), "unit": "GB/s",
                      "cores": 1, "kind": "oracle",
                      "sample": f"{len(times)} one-sequence append + decode steps, cycling "
                                f"through a seeded 48-sequence sample of the 70B-shape batch "
                                f"(log-uniform [128, 8192] tokens), fp64 oracle, "
                                f"{blas_threads()} BLAS thread(s), {sum(times):.1f} s",
                      "seconds": round(sum(times), 2), "host_cpus": os.cpu_count()}))


def blas_threads() -> str:
    return os.environ.get("OPENBLAS_NUM_THREADS", "default")


def single_thread_env(threads: int = 1):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
              "NUMEXPR_NUM_THREADS"):
        env[k] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def prefill_cpu_baseline_child(seed: int, budget_s: float) -> None:
    print(json.dumps(prefill_cpu_baseline(seed, budget_s)))


def cpu_baseline_subprocess(args):
    """The oracle with one BLAS thread (the reported value), and again with a
    BLAS thread per host core (reported beside it)."""
    child = "prefill_cpu_baseline_child" if args.workload == "prefill" else "cpu_baseline_child"
    code = ("import bench; bench.%s(%d, %f)" % (child, args.seed, args.cpu_seconds))

    def run(threads):
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT,
                           env=single_thread_env(threads), capture_output=True, text=True,
                           timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    try:
        out = run(1)
    except Exception as e:  # reported, not fatal: the GPU number stands on its own
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"failed: {type(e).__name__}: {e}"}
    threads = os.cpu_count() or 1
    try:
        allc = run(threads)
        out["all_threads"] = {"value": allc["value"], "threads": threads,
                              "sample": allc["sample"]}
    except Exception as e:
        out["all_threads"] = {"value": None, "threads": threads,
                              "sample": f"failed: {type(e).__name__}: {e}"}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if os.environ.get("OPENBLAS_NUM_THREADS") != "1":   # one BLAS thread, set before numpy loads
        os.execve(sys.executable, [sys.executable] + sys.argv, single_thread_env())
    case = oracle_sample_case(args.seed)
    oracle_steps(case, 0, max_steps=max(args.warmup, 0) or 1)
    times, nbytes = oracle_steps(case, 0, max_steps=args.steps)
    total = sum(times)
    value = sum(nbytes) / total / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe("cb70b") + " (oracle: one sequence per step, cycling a "
                                                   "48-sequence sample)", "batch": case.batch},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} steps of one sequence each from a 48-sequence "
                                   f"sample of the 70B-shape batch"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
# the copy-on-write step (prefix cache + pa_copy_blocks)
# ---------------------------------------------------------------------------

COW_METRIC = "copy-on-write block copy GB/s (bytes read + written), forked batch"
PREFILL_METRIC = "chunked-prefill paged attention TFLOP/s, 70B shape"


def cow_cpu_baseline(batch: int, block_elems: int, budget_s: float):
    """The oracle's block copy on the host (NumPy, one thread) over the same
    kind of step: `batch` 32 KiB K and V block copies per step."""
    import numpy as np
    from oracle import prefix_cache as pc
    nb = 1 + 2 * batch
    k = np.zeros((nb, block_elems), dtype=np.uint16)
    v = np.zeros_like(k)
    pairs = [(1 + i, 1 + batch + i) for i in range(batch)]
    steps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s or steps < 3:
        pc.copy_blocks(k, v, pairs)
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": round(4 * batch * block_elems * 2 * steps / dt / 1e9, 3), "unit": "GB/s",
            "cores": 1, "kind": "oracle",
            "sample": f"{steps} steps of {batch} K+V block copies (oracle copy_blocks, NumPy, "
                      f"blocks reused: host-cache resident), {dt:.1f} s"}


def run_cow(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    from paged_kv_cache_45_gb300 import binding as b

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    B, bs, hkv, d, sets = args.batch, 16, 8, 128, 32
    block_elems = bs * hkv * d
    block_bytes = block_elems * 2
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cow_cpu_baseline(B, block_elems, min(args.cpu_seconds, 5.0))

    # device pool and copy sets: every step copies B fresh blocks; 32 disjoint
    # sets (1 GiB of K+V) cycle, so a set's blocks are out of the L2 when reused
    nb = 1 + 2 * B * sets
    k_cache = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device=device)
    v_cache = torch.zeros_like(k_cache)
    rng = np.random.default_rng(args.seed + rank)
    ids = rng.permutation(np.arange(1, nb)).astype(np.int32).reshape(sets, 2, B)
    src = [torch.from_numpy(ids[i, 0].copy()).to(device) for i in range(sets)]
    dst = [torch.from_numpy(ids[i, 1].copy()).to(device) for i in range(sets)]
    stream = torch.cuda.current_stream(device)
    for w in range(args.warmup):
        b.pa_copy_blocks(k_cache, v_cache, src[w % sets], dst[w % sets])
    torch.cuda.synchronize()
    K = args.steps
    t_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.__enter__()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_ev[0].record(stream)
    for k in range(K):
        b.pa_copy_blocks(k_cache, v_cache, src[k % sets], dst[k % sets])
    t_ev[1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if sampler:
        sampler.__exit__(None, None, None)
    total_s = t_ev[0].elapsed_time(t_ev[1]) / 1e3
    step_bytes = 4 * B * block_bytes                  # K and V, read and written
    # the roofline's kernel duration: KI launches replayed from one CUDA graph
    # (a launch takes a few microseconds of device time, less than the host
    # needs to issue one, so directly issued launches leave the GPU idle in
    # between and per-launch events would time the host)
    KI = min(K, 256)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        b.pa_copy_blocks(k_cache, v_cache, src[0], dst[0])   # set-up outside the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            for k in range(KI):
                b.pa_copy_blocks(k_cache, v_cache, src[k % sets], dst[k % sets])
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    graph.replay()                                     # warm
    torch.cuda.synchronize()
    g_ev[0].record(stream)
    graph.replay()
    g_ev[1].record(stream)
    torch.cuda.synchronize()
    kern_s = g_ev[0].elapsed_time(g_ev[1]) / 1e3 / KI
    del graph

    # end to end through the public API: the host prefix cache forks the batch,
    # the children's first append asks for the copies, the pairs go to the
    # device, the kernel copies; the children are then discarded (host)
    pcache = b.PrefixCache(nb, bs)
    parents = []
    for i in range(B):
        sid, cached = pcache.admit(list(range(i * 1000, i * 1000 + 3 * bs + 5)))
        pcache.write_slots(sid, cached, 3 * bs + 5)
        parents.append(sid)
    E = min(args.e2e_steps, K)
    pin_src = torch.empty(B, dtype=torch.int32, pin_memory=True)
    pin_dst = torch.empty(B, dtype=torch.int32, pin_memory=True)
    dsrc = torch.empty(B, dtype=torch.int32, device=device)
    ddst = torch.empty(B, dtype=torch.int32, device=device)
    e2e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    e2e_ev[0].record(stream)
    for k in range(E):
        kids = pcache.fork_batch(parents)
        _, (cs, cd) = pcache.append_tokens(kids)
        stream.synchronize()                          # the pinned buffers are reused
        pin_src.numpy()[:] = cs
        pin_dst.numpy()[:] = cd
        dsrc.copy_(pin_src, non_blocking=True)
        ddst.copy_(pin_dst, non_blocking=True)
        b.pa_copy_blocks(k_cache, v_cache, dsrc, ddst)
        pcache.discard(kids)
    e2e_ev[1].record(stream)
    torch.cuda.synchronize()
    e2e_s = e2e_ev[0].elapsed_time(e2e_ev[1]) / 1e3
    stats = torch.tensor([total_s, step_bytes * K, e2e_s, step_bytes * E], dtype=torch.float64,
                         device=device)
    if world > 1:
        total_s, all_bytes, e2e_s, e2e_bytes = combine_ranks(stats)
    else:
        all_bytes, e2e_bytes = step_bytes * K, step_bytes * E
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_hbm_peak()
    gbs = all_bytes / total_s / 1e9
    kern_gbs = step_bytes / kern_s / 1e9
    line = {
        "metric": COW_METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_s / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes)",
        "data": "synthetic (zero-filled pool; seeded block ids)",
        "config": {"workload": describe("cow", B), "batch": B, "block_bytes": block_bytes,
                   "l2": "32 disjoint copy sets (1 GiB) cycled: each set is out of the 129 MB "
                         "L2 when it comes round again",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_peak": round(100 * gbs / peak, 2),
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel", "achieved": round(kern_gbs, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(kern_gbs / peak, 4),
                     "peak_kind": f"{peak_kind} hbm_gbs (a copy: bytes read + written)",
                     "traffic": None, "algorithmic_bytes_per_launch": step_bytes,
                     "measured": f"CUDA events around a CUDA-graph replay of {KI} launches "
                                 f"(device time a launch; the directly issued steps above "
                                 f"are bound by the host's issue rate)"},
        "e2e": {"value": round(e2e_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 0, "steps": E,
                "note": "host prefix cache fork + append (decides the copies), H2D of the "
                        "pairs, copy kernel, host discard; the result stays in the pool"},
        "gpu_launches": K,
        "source_sha16": library_source_hash(),
        "timing": "CUDA events bracketing the K steps on the launching stream",
    }
    if sampler:
        line["clocks"] = sampler.summary()
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "cow":
        run_cow(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
