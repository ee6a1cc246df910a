#!/usr/bin/env python3
"""Benchmark of one paged decode-attention step on GB300.

A step is one attention layer's decode step for the whole batch: the new
tokens' K/V written into the paged cache (reshape_and_cache or quantize_kv),
attention over every sequence's visible tokens, and the log-sum-exp reduce
where the schedule splits.  The decode workloads run the step as one launch
(pkv_decode_step_balanced: write + balanced attention); --schedule picks
another.  The headline workload is the Llama-3-8B-like batch (batch 8, 32/8
heads, head_dim 128, bf16, ragged contexts 512..4096).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  `value` is algorithmic bytes (K + V + q + out +
block tables + the write's bytes) per second of device time over the K timed
steps; inputs are resident in HBM and rotate over enough replicas that the
bytes touched between two uses of one replica exceed the L2 cache.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
L2_BYTES_FALLBACK = 126 * 2 ** 20
METRIC = "paged-decode attention KV-read GB/s (% of HBM peak); decode steps/sec"

WORKLOADS = {
    "tiny_f16": 1,
    "llama3_8b_batch8": 2,
    "long_context_32k": 3,
    "k8v4_batch32": 4,
    "verify_batch256": 5,
    "sliding_window_b8_w4096": "sliding_window_b8_w4096",
    "cascade_b32_p2048": "cascade_b32_p2048",
    "sparse_b4_32k": "sparse_b4_32k",
}
DEFAULT_WORKLOAD = "llama3_8b_batch8"
# schedule of the attention call per workload: the 32K workload is defined with
# fixed 512-token partitions and a separate reduce; the decode ones run the whole
# step (cache write + balanced attention) as one launch (the tiny one too: 4.3 us
# against 5.2 us for write + single pass, launch-bound); the verify batch keeps
# the write as its own launch (measured a little faster); the shared-prompt and
# sparse workloads run their own entry points
DEFAULT_SCHEDULE = {"tiny_f16": "fused", "llama3_8b_batch8": "fused", "long_context_32k": "split",
                    "k8v4_batch32": "fused", "verify_batch256": "balanced",
                    "sliding_window_b8_w4096": "fused", "cascade_b32_p2048": "cascade",
                    "sparse_b4_32k": "sparse"}
KERNEL_NAME = {"single": "pkv_paged_attention", "split": "pkv_paged_attention_split",
               "balanced": "pkv_paged_attention_balanced", "fused": "pkv_decode_step_balanced",
               "cascade": "pkv_paged_attention_cascade", "sparse": "pkv_paged_attention_sparse"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--partition", type=int, default=None, help="split-KV partition size (with --schedule split)")
    ap.add_argument("--schedule", default=None,
                    choices=["single", "split", "balanced", "fused", "cascade", "sparse"],
                    help="attention schedule (default: per workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle sample budget")
    ap.add_argument("--quick", action="store_true",
                    help="no clock hold, e2e or CPU baseline (for profiler runs)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_bandwidth_gbs"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (ms) over the process group, when
    there is one with more than one rank; the job's time is its slowest rank's."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world_size, bytes_per_rank_step, ms_per_step):
    """Whole-job GB/s: every rank moved its own step's bytes in the (max) step time."""
    return world_size * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def make_workload(name, device, seed_offset=0, partition=None):
    from paged_decode_attention_cache_gb300 import workloads as W
    key = WORKLOADS[name]
    fn = W.CONFIGS[key] if isinstance(key, int) else W.EXTRA[key]
    kw = {}
    if partition is not None and name != "tiny_f16":
        kw["partition_size"] = partition
    import inspect
    sig = inspect.signature(fn)
    seed = sig.parameters["seed"].default + seed_offset
    w = fn(device=device, seed=seed, **kw) if "partition_size" in sig.parameters else fn(device=device, seed=seed)
    if name == "tiny_f16" and partition is not None:
        w.partition_size = partition
    return w


def step_bytes(w, cascade_plan=None, sparse=False):
    """(attention bytes, write bytes) of one step; cascade_plan = (members,
    item_blocks) counts each item's shared prefix once; sparse counts only the
    listed pages."""
    from paged_decode_attention_cache_gb300 import bytes_model as BM
    ctx = [int(c) for c in w.context_lens.cpu()]
    if sparse:
        attn = BM.sparse_attention_bytes(ctx, w.page_lists.cpu().tolist(), w.page_counts.cpu().tolist(),
                                         w.num_heads, w.num_kv_heads, w.head_dim, w.cache)
    elif cascade_plan is not None:
        members, blocks = (x.cpu().tolist() for x in cascade_plan)
        attn = BM.cascade_attention_bytes(ctx, members, blocks, w.num_heads, w.num_kv_heads, w.head_dim, w.cache)
    else:
        attn = BM.attention_bytes(ctx, w.q_len, w.num_heads, w.num_kv_heads, w.head_dim, w.cache,
                                  sliding_window=w.sliding_window)
    wr = BM.write_bytes(int(w.slot_new.numel()), w.num_kv_heads, w.head_dim, w.cache)
    return attn, wr


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_decode_attention_cache_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profiles(workload, kernel):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel sources (null otherwise)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        e = d.get(f"{kernel}:{workload}")
        if e and e.get("source_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        import tempfile
        # the raw samples: a scratch file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"pkv_clocks_{os.getpid()}.csv")
        self.device_index = device_index

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.device_index), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(w, attn_bytes, budget_s, split=False, sparse=False):
    """The oracle as it stands, on this host's cores, over whole steps of the
    same workload until the time budget is spent (at least one step)."""
    import numpy as np  # noqa: F401
    from tests.helpers import oracle_attention, oracle_cache_after_step
    threads = os.cpu_count() or 1
    cs = oracle_cache_after_step(w)
    import oracle
    split = split and w.partition_size > 0
    n, t0 = 0, time.perf_counter()
    while True:
        if sparse:   # only the listed pages
            oracle_attention(w, cs, threads=threads, sparse=True)
        elif split:   # phase 1 partials, then the LSE reduce, as the GPU step does
            _, part = oracle_attention(w, cs, threads=threads, partition_size=w.partition_size,
                                       max_partitions=w.max_partitions, want_out=False)
            oracle.lse_reduce(*part)
        else:
            oracle_attention(w, cs, threads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el / n * (n + 1) > 3 * budget_s:
            break
    per = el / n
    return {"value": attn_bytes / per / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full attention step(s) of {w.name} (fp64 scalar oracle"
                      + (": the listed pages only" if sparse else ": split-KV partials + LSE reduce" if split else "")
                      + f"), {per:.3f} s each", "seconds_per_step": per}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = make_workload(args.workload, "cpu", 0, args.partition)
    schedule = args.schedule or DEFAULT_SCHEDULE[args.workload]
    plan = None
    if schedule == "cascade":   # bytes as the GPU arm counts them (the oracle itself is plain attention)
        from paged_decode_attention_cache_gb300 import build as pkv_build, ops
        from paged_decode_attention_cache_gb300.runner import cascade_plan_for
        pkv_build.build()
        plan = cascade_plan_for(w)
    attn_b, wr_b = step_bytes(w, plan, sparse=(schedule == "sparse"))
    cb = cpu_baseline(w, attn_b + wr_b, max(1.0, min(args.cpu_seconds, 20.0)), split=(schedule == "split"),
                      sparse=(schedule == "sparse"))
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["seconds_per_step"] * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name},
            "cpu_baseline": {k: cb[k] for k in ("kind", "cores", "sample", "value", "unit")},
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    from paged_decode_attention_cache_gb300 import build as pkv_build, ops
    from paged_decode_attention_cache_gb300.runner import DecodeStep
    if rank == 0 or ws == 1:
        pkv_build.build()
    if ws > 1:
        torch.distributed.barrier()
    ops.lib()

    w = make_workload(args.workload, dev, seed_offset=rank, partition=args.partition)
    schedule = args.schedule or DEFAULT_SCHEDULE[args.workload]
    if args.partition is not None and args.schedule is None:
        schedule = "split" if args.partition > 0 else "single"
    if schedule == "split" and w.partition_size <= 0:
        w.partition_size = 512
    first = DecodeStep(w, dev, schedule=schedule)
    plan = (first.members, first.item_blocks) if schedule == "cascade" else None
    attn_b, wr_b = step_bytes(w, plan, sparse=(schedule == "sparse"))
    total_b = attn_b + wr_b
    l2 = getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0) or L2_BYTES_FALLBACK
    reps = max(2, math.ceil(3 * l2 / max(1, total_b)))
    reps = min(reps, 16)
    steps_ = [first] + [DecodeStep(w, dev, schedule=schedule) for _ in range(reps - 1)]
    launches = steps_[0].launches_per_step()

    for i in range(max(3, args.warmup)):
        steps_[i % reps].step()
    torch.cuda.synchronize()
    # The timed steps replay CUDA graphs: one graph holds `n_cycle` consecutive
    # steps over the rotating replicas, so host launch overhead stays off the
    # device timeline.  A second graph holds the same number of launches of the
    # dominant kernel alone, for its average duration.
    U = max(1, math.ceil(64 / reps))
    n_cycle = U * reps
    cycle, attn_only = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    singles = [torch.cuda.CUDAGraph() for _ in range(reps)]
    with torch.cuda.graph(cycle):
        for _ in range(U):
            for st in steps_:
                st.step()
    with torch.cuda.graph(attn_only):
        for _ in range(U):
            for st in steps_:
                st.attend_phase1()
    for st, gph in zip(steps_, singles):
        with torch.cuda.graph(gph):
            st.step()
    stream = torch.cuda.current_stream()
    cycle.replay()
    attn_only.replay()
    torch.cuda.synchronize()
    # hold the clocks under load for a moment so the sampler sees the loaded state
    sampler = ClockSampler(local)
    if not args.quick:
        sampler.start()
    t_end = time.perf_counter() + (0.0 if args.quick else 1.0)
    while time.perf_counter() < t_end:
        for _ in range(20):
            cycle.replay()
        torch.cuda.synchronize()

    K = args.steps
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(K // n_cycle):
        cycle.replay()
    for k in range(K % n_cycle):
        singles[k % reps].replay()
    stop.record(stream)
    torch.cuda.synchronize()
    step_ms = start.elapsed_time(stop) / K
    # dominant kernel: back-to-back launches (rotating replicas), inside the loaded window
    n_attn = max(1, K // n_cycle)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_attn):
        attn_only.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if not args.quick else None
    kern_ms = a0.elapsed_time(a1) / (n_attn * n_cycle)
    step_ms, kern_ms = max_over_ranks([step_ms, kern_ms], dev)
    flags = 0
    for st in steps_:
        flags |= st.error_flags()

    # end to end through the same API with host buffers: pinned inputs copied in,
    # the output copied back, every step
    e2e = None
    if not (args.no_e2e or args.quick):
        st = steps_[0]
        # the step's inputs packed in one pinned host buffer, copied with one
        # host-to-device transfer into one device buffer whose views the step
        # reads; the output comes back with one device-to-host transfer
        src = [st.q, st.k_new, st.v_new, st.slot_new, st.seqs.block_tables, st.seqs.context_lens]
        if schedule == "cascade":
            src += [st.members, st.item_blocks]
        if schedule == "sparse":
            src += [st.page_lists, st.page_counts]
        offs, total = [], 0
        for x in src:
            offs.append(total)
            total += (x.numel() * x.element_size() + 255) // 256 * 256
        host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
        views = []
        for x, o in zip(src, offs):
            n = x.numel() * x.element_size()
            host_buf[o:o + n].copy_(x.contiguous().view(-1).view(torch.uint8).cpu())
            views.append(dev_buf[o:o + n].view(x.dtype).view(x.shape))
        st.q, st.k_new, st.v_new, st.slot_new, st.seqs.block_tables, st.seqs.context_lens = views[:6]
        if schedule == "cascade":
            st.members, st.item_blocks = views[6:]
        if schedule == "sparse":
            st.page_lists, st.page_counts = views[6:]
        host_out = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
        h2d = total
        d2h = host_out.numel() * host_out.element_size()
        Ke = max(10, min(K, 500))
        for _ in range(3):
            dev_buf.copy_(host_buf, non_blocking=True)
            st.step()
            host_out.copy_(st.out, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            dev_buf.copy_(host_buf, non_blocking=True)
            st.step()
            host_out.copy_(st.out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / Ke
        e2e_ms = max_over_ranks([e2e_ms], dev)[0]
        e2e = {"value": job_throughput(ws, total_b, e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    peak, peak_src = load_peaks()
    # the fused decode step's kernel also writes the new tokens
    kern_b = attn_b + (wr_b if schedule == "fused" else 0)
    achieved = kern_b / (kern_ms * 1e-3) / 1e9
    kernel_name = KERNEL_NAME[schedule]
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic_from_profiles(w.name, kernel_name), "kernel": kernel_name,
                "kernel_ms": kern_ms, "peak_source": f"{peak_src} (copy bandwidth)",
                "frac_of_nominal_8000": achieved / 8000.0}
    cb = None
    if rank == 0 and not (args.no_cpu_baseline or args.quick):
        wc = make_workload(args.workload, "cpu", 0, args.partition)
        cb = cpu_baseline(wc, total_b, args.cpu_seconds, split=(schedule == "split"), sparse=(schedule == "sparse"))
        cb.pop("seconds_per_step", None)

    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return 0
    value = job_throughput(ws, total_b, step_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.num_seqs, "q_len": w.q_len, "heads": w.num_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "cache": w.cache,
                   "schedule": schedule, "partition_size": steps_[0].partition_size,
                   "sum_context": int(w.context_lens.sum()),
                   **({"cascade_items": int(first.members.shape[0]),
                       "plain_attention_bytes": step_bytes(w)[0]} if schedule == "cascade" else {}),
                   **({"pages_listed": int(w.page_counts.sum()),
                       "dense_attention_bytes": step_bytes(w)[0]} if schedule == "sparse" else {}),
                   "bytes_per_step": total_b, "parallelism": f"replicas x{ws}",
                   "l2": f"{reps} rotating input replicas, {reps * total_b / 2**20:.0f} MiB touched per cycle "
                         f"vs {l2 / 2**20:.0f} MiB L2"},
        "steps_per_s": 1e3 / step_ms * ws,
        "tokens_per_s": 1e3 / step_ms * ws * w.num_seqs * w.q_len,
        "roofline": roofline,
        "cpu_baseline": cb,
        "e2e": e2e,
        "gpu_launches": K * launches,
        "clocks": clocks,
        "device_error_flags": flags,
    }
    print(json.dumps(line))
    return 0 if flags == 0 else 3


if __name__ == "__main__":
    sys.exit(main())
