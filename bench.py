#!/usr/bin/env python3
"""Benchmark of the paged decode-attention step on GB300.

A step is one attention layer's decode step for the whole batch: the new
tokens' K/V written into the paged cache (reshape_and_cache or quantize_kv),
attention over every sequence's visible tokens, and the log-sum-exp reduce
where the schedule splits.  The decode workloads run the step as one launch
(pkv_decode_step_balanced: write + balanced attention); --schedule picks
another.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats R] [--workload NAME]
                  [--impl reference] [--quick]

Prints one JSON line (rank 0).  The headline (`value`, `ms_per_step`,
`roofline`, `e2e`) is the Llama-3-8B-like batch (batch 8, 32/8 heads, head_dim
128, bf16, ragged contexts 512..4096): the metric names no workload, and this
is the decode step it is phrased for.  `per_config` holds the same
measurements for all five workloads of the set (tiny fp16, the Llama-3-8B-like
batch, 32K split-KV, K8/V4 batch 32, verify batch 256).

Timing.  Inputs are resident in HBM.  Each measurement is EXACTLY K back-to-back
steps, captured as CUDA graphs (at most 1000 steps per graph) over enough
replicas of the whole workload (pools included) that the bytes touched between
two uses of one replica exceed 3x the L2 size; a spin kernel before the start
event keeps the GPU busy while the host enqueues the graphs, so no host gap is
timed.  The measurement is repeated R times (CUDA events on the replay stream,
barrier + synchronize around each, max over ranks) and the median is reported
with p10 / p90.  `value` = algorithmic bytes (K + V + q + out + block tables +
the write's bytes) per second of the median step.  The dominant kernel is timed
the same way, alone (`kernel_ms`); `roofline.achieved` is its algorithmic bytes
per launch / its median duration.  A hot-L2 figure (one replica, back to back)
is reported beside each, labelled.
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
GRAPH_MAX_STEPS = 1000
SLEEP_CYCLES = 400_000   # ~0.2 ms of spinning ahead of each timed region

WORKLOADS = ["tiny_f16", "llama3_8b_batch8", "long_context_32k", "k8v4_batch32", "verify_batch256",
             "sliding_window_b8_w4096", "cascade_b32_p2048", "sparse_b4_32k"]
# the five decode / verify workloads reported in per_config
CONFIG_ORDER = ["tiny_f16", "llama3_8b_batch8", "long_context_32k", "k8v4_batch32", "verify_batch256"]
DEFAULT_WORKLOAD = "llama3_8b_batch8"
# schedule of the attention call per workload: the decode ones run the whole
# step (cache write + balanced attention) as one launch (the tiny one too:
# launch-bound, one launch beats two); the 32K workload runs split-KV with the
# log-sum-exp combine fused (balanced cost ranges as the partitions), and its
# fixed 512-token partitions + separate reduce are timed beside it (ALT_SCHEDULE);
# the verify batch keeps the write as its own launch (measured a little faster);
# the shared-prompt and sparse workloads run their own entry points
DEFAULT_SCHEDULE = {"tiny_f16": "fused", "llama3_8b_batch8": "fused", "long_context_32k": "balanced",
                    "k8v4_batch32": "fused", "verify_batch256": "balanced",
                    "sliding_window_b8_w4096": "fused", "cascade_b32_p2048": "cascade",
                    "sparse_b4_32k": "sparse"}
ALT_SCHEDULE = {"long_context_32k": "split"}
KERNEL_NAME = {"single": "pkv_paged_attention", "split": "pkv_paged_attention_split",
               "balanced": "pkv_paged_attention_balanced", "fused": "pkv_decode_step_balanced",
               "cascade": "pkv_paged_attention_cascade", "sparse": "pkv_paged_attention_sparse"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--repeats", type=int, default=7, help="timed repetitions of the K steps (median, p10, p90)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--partition", type=int, default=None, help="split-KV partition size (with --schedule split)")
    ap.add_argument("--schedule", default=None,
                    choices=["single", "split", "balanced", "fused", "cascade", "sparse"],
                    help="attention schedule of the headline workload (default: per workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="headline workload only (no per_config)")
    ap.add_argument("--cpu-seconds", type=float, default=3.0, help="oracle time budget per baseline leg")
    ap.add_argument("--quick", action="store_true",
                    help="headline only: no per_config, clocks, e2e or CPU baseline (for profiler runs)")
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


def summary(times):
    """(median, p10, p90) of a list of per-step times."""
    xs = sorted(times)
    if len(xs) == 1:
        return xs[0], xs[0], xs[0]

    def pct(p):
        k = (len(xs) - 1) * p
        lo = int(math.floor(k))
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)

    return statistics.median(xs), pct(0.1), pct(0.9)


def make_workload(name, device, seed_offset=0, partition=None):
    from paged_decode_attention_cache_gb300 import workloads as W
    fn = W.BY_NAME[name]
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


def step_bytes(w, cascade_plan=None, sparse=False, seqs=None):
    """(attention bytes, write bytes) of one step; cascade_plan = (members,
    item_blocks) counts each item's shared prefix once; sparse counts only the
    listed pages; seqs restricts the count to those sequences (no write)."""
    from paged_decode_attention_cache_gb300 import bytes_model as BM
    ctx = [int(c) for c in w.context_lens.cpu()]
    if seqs is not None:
        ctx = [ctx[s] for s in seqs]
    if sparse:
        pl, pc = w.page_lists.cpu().tolist(), w.page_counts.cpu().tolist()
        if seqs is not None:
            pl, pc = [pl[s] for s in seqs], [pc[s] for s in seqs]
        attn = BM.sparse_attention_bytes(ctx, pl, pc, w.num_heads, w.num_kv_heads, w.head_dim, w.cache)
    elif cascade_plan is not None and seqs is None:
        members, blocks = (x.cpu().tolist() for x in cascade_plan)
        attn = BM.cascade_attention_bytes(ctx, members, blocks, w.num_heads, w.num_kv_heads, w.head_dim, w.cache)
    else:
        attn = BM.attention_bytes(ctx, w.q_len, w.num_heads, w.num_kv_heads, w.head_dim, w.cache,
                                  sliding_window=w.sliding_window)
    if seqs is not None:
        return attn, 0
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
        try:
            os.unlink(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU timing

def capture_steps(fn, K):
    """CUDA graphs holding exactly K calls fn(k), k = 0..K-1, at most
    GRAPH_MAX_STEPS per graph (replayed back to back)."""
    import torch
    graphs, k = [], 0
    while k < K:
        n = min(GRAPH_MAX_STEPS, K - k)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(k, k + n):
                fn(i)
        graphs.append(g)
        k += n
    return graphs


def time_graphs(graphs, K, R, device, ws):
    """R timed runs of the graphs back to back (exactly K steps each): per-step
    ms of every run, max over ranks."""
    import torch
    stream = torch.cuda.current_stream()
    for g in graphs:   # untimed pass
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(R):
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(SLEEP_CYCLES)   # the GPU is busy while the host enqueues the graphs
        e0.record(stream)
        for g in graphs:
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / K)
    return max_over_ranks(times, device)


def cold_step_times(step, n, device):
    """Per-step ms of n eager steps, each after an L2 flush (a write larger than
    L2); the step's launches are enqueued while the flush runs."""
    import torch
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or L2_BYTES_FALLBACK
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    out = []
    for _ in range(n):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


class Bench:
    """One workload on this GPU: its replicas, graphs and measurements."""

    def __init__(self, name, schedule, partition, dev, rank, ws):
        import torch
        from paged_decode_attention_cache_gb300.runner import DecodeStep
        self.name, self.dev, self.ws = name, dev, ws
        w = make_workload(name, dev, seed_offset=rank, partition=partition)
        if schedule is None:
            schedule = DEFAULT_SCHEDULE[name]
            if partition is not None:
                schedule = "split" if partition > 0 else "single"
        if schedule == "split" and w.partition_size <= 0:
            w.partition_size = 512
        self.w, self.schedule = w, schedule
        first = DecodeStep(w, dev, schedule=schedule)
        self.plan = (first.members, first.item_blocks) if schedule == "cascade" else None
        self.attn_b, self.wr_b = step_bytes(w, self.plan, sparse=(schedule == "sparse"))
        self.total_b = self.attn_b + self.wr_b
        # the fused decode step's kernel also writes the new tokens
        self.kern_b = self.attn_b + (self.wr_b if schedule == "fused" else 0)
        idx = torch.device(dev).index or 0
        self.l2 = getattr(torch.cuda.get_device_properties(idx), "L2_cache_size", 0) or L2_BYTES_FALLBACK
        self.reps = min(16, max(2, math.ceil(3 * self.l2 / max(1, self.total_b))))
        self.steps = [first] + [DecodeStep(w, dev, schedule=schedule) for _ in range(self.reps - 1)]
        self.launches = first.launches_per_step()
        self.partition_size = first.partition_size

    def l2_note(self):
        touched = self.reps * self.total_b
        if touched >= 3 * self.l2:
            return (f"{self.reps} rotating input replicas, {touched / 2**20:.0f} MiB touched per cycle vs "
                    f"{self.l2 / 2**20:.0f} MiB L2 (inputs larger than L2)")
        return (f"L2-resident: the whole workload ({self.reps} replicas, {touched / 2**20:.1f} MiB) fits in the "
                f"{self.l2 / 2**20:.0f} MiB L2; cold_l2 flushes L2 before each step")

    def run(self, K, W, R, hot=True):
        import torch
        st = self.steps
        reps = self.reps
        for i in range(max(3, W)):
            st[i % reps].step()
        torch.cuda.synchronize()
        step_g = capture_steps(lambda k: st[k % reps].step(), K)
        self.step_t = time_graphs(step_g, K, R, self.dev, self.ws)
        del step_g
        if self.launches == 1 and self.schedule != "split":
            self.kern_t = self.step_t   # the step is the dominant kernel's single launch
        else:
            kern_g = capture_steps(lambda k: st[k % reps].attend_phase1(), K)
            self.kern_t = time_graphs(kern_g, K, R, self.dev, self.ws)
            del kern_g
        self.hot_t = None
        if hot:
            hot_g = capture_steps(lambda k: st[0].step(), K)
            self.hot_t = time_graphs(hot_g, K, R, self.dev, self.ws)
            del hot_g
        self.flags = 0
        for s in st:
            self.flags |= s.error_flags()

    def result(self, peak, peak_src):
        med, p10, p90 = summary(self.step_t)
        kmed, kp10, kp90 = summary(self.kern_t)
        w, ws = self.w, self.ws
        achieved = self.kern_b / (kmed * 1e-3) / 1e9
        kernel = KERNEL_NAME[self.schedule]
        r = {
            "workload": w.name, "schedule": self.schedule, "batch": w.num_seqs, "q_len": w.q_len,
            "heads": w.num_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "cache": w.cache,
            "partition_size": self.partition_size, "sum_context": int(w.context_lens.sum()),
            "bytes_per_step": self.total_b, "launches_per_step": self.launches, "l2": self.l2_note(),
            "ms_per_step": med, "ms_per_step_p10": p10, "ms_per_step_p90": p90,
            "value": job_throughput(ws, self.total_b, med), "unit": "GB/s",
            "steps_per_s": 1e3 / med * ws, "tokens_per_s": 1e3 / med * ws * w.num_seqs * w.q_len,
            "kernel": kernel, "kernel_ms": kmed, "kernel_ms_p10": kp10, "kernel_ms_p90": kp90,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic_from_profiles(w.name, kernel),
                         "kernel_bytes_per_launch": self.kern_b,
                         "peak_source": f"{peak_src} (copy bandwidth)"},
            "device_error_flags": self.flags,
        }
        if self.hot_t is not None:
            hmed, _, _ = summary(self.hot_t)
            r["hot_l2"] = {"ms_per_step": hmed, "value": job_throughput(ws, self.total_b, hmed),
                           "note": "one replica stepped back to back: its cache stays partly in L2"}
        return r

    def free(self):
        import torch
        self.steps = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def e2e_measure(bench, K, device, ws):
    """The same step through the public API with host buffers, run as a serving
    loop runs it: every step's inputs are packed in a pinned host buffer and
    copied in with one host-to-device transfer, the step is launched, and its
    output is copied back to pinned host memory.  Independent replicas (request
    groups) are served in two banks of G that alternate, so one bank's copies
    overlap the other bank's kernels: a bank's G copies in on one stream, its G
    steps back to back on the capture stream, their copies out on a third;
    events put a bank's steps after its inputs' copies and after the copies out
    of its previous steps, and its copies in after its previous steps.  Only
    the first step of a bank waits on a copy: a kernel that depends on a copy
    is not launched under the previous kernel's tail (programmatic dependent
    launch), so each wait costs a step the full grid-completion hop.  The loop
    is captured in CUDA graphs like the device-timed steps (eager launches
    would time the host's enqueue rate instead)."""
    import torch
    from paged_decode_attention_cache_gb300.runner import DecodeStep
    # replicas per bank: 4 when eight copies of the step's data stay small (extra
    # replicas are made for it), else as many as the device-timed rotation holds
    G = 4 if 8 * bench.total_b <= (1 << 31) else max(1, min(4, bench.reps // 2))
    NR = 2 * G
    steps = list(bench.steps[:NR]) + [DecodeStep(bench.w, device, schedule=bench.schedule)
                                      for _ in range(NR - min(NR, bench.reps))]
    pairs = []
    for r in range(NR):
        st = steps[r]
        schedule = bench.schedule
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
        dev_buf = torch.empty(total, dtype=torch.uint8, device=device)
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
        pairs.append((st, host_buf, dev_buf, host_out))
    h2d = pairs[0][2].numel()
    d2h = pairs[0][3].numel() * pairs[0][3].element_size()
    Ke = max(2 * NR, min(K, 500)) // NR * NR   # whole cycles of both banks
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(cap)
            h2d_s.wait_event(fork)
            d2h_s.wait_event(fork)
            ev_in = [torch.cuda.Event() for _ in range(2)]
            ev_done = [torch.cuda.Event() for _ in range(2)]
            ev_out = [torch.cuda.Event() for _ in range(2)]
            nb = n // G
            for j in range(nb):
                b = j & 1
                bank = pairs[b * G:(b + 1) * G]
                if j >= 2:
                    h2d_s.wait_event(ev_done[b])   # the bank's previous steps have read these buffers
                with torch.cuda.stream(h2d_s):
                    for st, hb, db, ho in bank:
                        db.copy_(hb, non_blocking=True)
                    ev_in[b].record(h2d_s)
                cap.wait_event(ev_in[b])
                if j >= 2:
                    cap.wait_event(ev_out[b])      # their outputs have been copied out
                for st, hb, db, ho in bank:
                    st.step(cap)
                ev_done[b].record(cap)
                d2h_s.wait_event(ev_done[b])
                with torch.cuda.stream(d2h_s):
                    for st, hb, db, ho in bank:
                        ho.copy_(st.out, non_blocking=True)
                    ev_out[b].record(d2h_s)
            cap.wait_event(ev_in[(nb - 1) & 1])
            cap.wait_event(ev_out[0])
            cap.wait_event(ev_out[1])
        return g

    per_graph = max(NR, GRAPH_MAX_STEPS // NR * NR)
    graphs = [capture(n) for n in [min(per_graph, Ke - k) for k in range(0, Ke, per_graph)]]
    times = time_graphs(graphs, Ke, 3, device, ws)
    e2e_ms = sorted(times)[len(times) // 2]
    return {"value": job_throughput(ws, bench.total_b, e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": Ke,
            "how": f"pinned host inputs copied in and the output copied back every step; two banks of {G} "
                   "independent replicas alternate so one bank's copies overlap the other's kernels, and "
                   "a bank's steps run back to back; captured in CUDA graphs"}


# ---------------------------------------------------------------- the oracle on the host

def oracle_step_time(w, schedule, seqs, threads, cache_state):
    """Seconds the oracle takes for attention over the listed sequences (split
    schedule: its partials, then the LSE reduce, as the GPU step does)."""
    import oracle
    from oracle import from_workload as OW
    rows = [s * w.q_len + j for s in seqs for j in range(w.q_len)]
    t0 = time.perf_counter()
    if schedule == "sparse":
        OW.attention(w, cache_state, rows=rows, threads=threads, sparse=True)
    elif schedule == "split" and w.partition_size > 0:
        _, part = OW.attention(w, cache_state, rows=rows, threads=threads, partition_size=w.partition_size,
                               max_partitions=w.max_partitions, want_out=False)
        oracle.lse_reduce(*part)
    else:
        OW.attention(w, cache_state, rows=rows, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, schedule, threads, budget_s, cache_state=None, seed=0):
    """The oracle as it stands, on `threads` host threads, over a bounded
    sample of the workload: the first n sequences of a seeded order, n grown
    until the sample takes about budget_s (the whole batch if it fits).
    value = algorithmic attention bytes of the sample / its time."""
    import random
    from oracle import from_workload as OW
    cs = cache_state or OW.cache_after_step(w)
    order = list(range(w.num_seqs))
    random.Random(seed).shuffle(order)
    n = 1
    t = oracle_step_time(w, schedule, order[:1], threads, cs)
    while n < w.num_seqs and t < budget_s:
        n2 = min(w.num_seqs, max(n + 1, int(n * min(8.0, 0.9 * budget_s / max(t, 1e-6)))))
        t = oracle_step_time(w, schedule, order[:n2], threads, cs)
        n = n2
    b, _ = step_bytes(w, sparse=(schedule == "sparse"), seqs=order[:n])
    what = ("the listed pages of " if schedule == "sparse" else
            "split-KV partials + LSE reduce over " if schedule == "split" and w.partition_size > 0 else "")
    sample = (f"attention over {what}{n} of {w.num_seqs} sequences of {w.name} (seeded order), "
              f"fp64 scalar oracle, {t:.3f} s")
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
            "seconds": t, "sample_bytes": b}


def cpu_baselines(w, schedule, budget_s):
    """Single-thread and all-core oracle times on the same workload."""
    from oracle import from_workload as OW
    cs = OW.cache_after_step(w)
    allc = os.cpu_count() or 1
    one = cpu_baseline(w, schedule, 1, budget_s, cs)
    many = cpu_baseline(w, schedule, allc, budget_s, cs)
    out = dict(many)
    out["single_thread"] = {"value": one["value"], "cores": 1, "sample": one["sample"]}
    return out


def run_reference(args):
    """The oracle as the reference arm: exactly K steps (after W untimed ones)
    of the headline workload on this host's cores, each step the whole batch's
    attention (split: partials + LSE reduce)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import from_workload as OW
    w = make_workload(args.workload, "cpu", 0, args.partition)
    schedule = args.schedule or DEFAULT_SCHEDULE[args.workload]
    if schedule == "split" and w.partition_size <= 0:
        w.partition_size = 512
    plan = None
    if schedule == "cascade":   # bytes as the GPU arm counts them (the oracle itself is plain attention)
        from paged_decode_attention_cache_gb300 import build as pkv_build
        from paged_decode_attention_cache_gb300.runner import cascade_plan_for
        pkv_build.build()
        plan = cascade_plan_for(w)
    attn_b, wr_b = step_bytes(w, plan, sparse=(schedule == "sparse"))
    threads = os.cpu_count() or 1
    cs = OW.cache_after_step(w)
    seqs = list(range(w.num_seqs))
    for _ in range(max(0, args.warmup)):
        oracle_step_time(w, schedule, seqs, threads, cs)
    times = [oracle_step_time(w, schedule, seqs, threads, cs) for _ in range(max(1, args.steps))]
    per = sum(times) / len(times)
    value = (attn_b + wr_b) / per / 1e9
    sample = (f"{len(times)} whole attention step(s) of {w.name} (fp64 scalar oracle"
              + (": the listed pages only" if schedule == "sparse" else
                 ": split-KV partials + LSE reduce" if schedule == "split" else "")
              + f"), {per:.3f} s each")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "schedule": schedule},
            "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": sample, "value": value, "unit": "GB/s"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- main

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
    if rank == 0 or ws == 1:
        pkv_build.build()
    if ws > 1:
        torch.distributed.barrier()
    ops.lib()
    K, W, R = max(1, args.steps), args.warmup, max(1, args.repeats)
    peak, peak_src = load_peaks()
    do_configs = not (args.quick or args.no_configs)
    do_cpu = rank == 0 and not (args.no_cpu_baseline or args.quick)

    sampler = ClockSampler(local)
    if not args.quick:
        sampler.start()
        # hold the clocks under load for a moment so the sampler sees the loaded state
        warm = Bench(args.workload, args.schedule, args.partition, dev, rank, ws)
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for i in range(50):
                warm.steps[i % warm.reps].step()
            torch.cuda.synchronize()
        warm.free()
        del warm

    head = Bench(args.workload, args.schedule, args.partition, dev, rank, ws)
    head.run(K, W, R, hot=not args.quick)
    head_res = head.result(peak, peak_src)
    e2e = None
    if not (args.no_e2e or args.quick):
        e2e = e2e_measure(head, K, dev, ws)

    per_config = {}
    kept = {}
    if do_configs:
        for name in CONFIG_ORDER:
            if name == args.workload and head.schedule == DEFAULT_SCHEDULE[name] and args.partition is None:
                b, res = head, dict(head_res)
            else:
                b = Bench(name, None, None, dev, rank, ws)
                b.run(K, W, R)
                res = b.result(peak, peak_src)
            if name == "tiny_f16":
                # launch-bound: also one graph of 1000 steps, and cold-L2 eager steps
                g = capture_steps(lambda k: b.steps[k % b.reps].step(), 1000)
                gt = time_graphs(g, 1000, R, dev, ws)
                del g
                res["graph_1000_steps"] = {"ms_per_step": summary(gt)[0],
                                           "note": "one CUDA graph of 1000 steps over the replicas"}
                cold = cold_step_times(b.steps[0].step, max(10, min(50, K)), torch.device(dev))
                cm, c10, c90 = summary(cold)
                res["cold_l2"] = {"ms_per_step": cm, "ms_per_step_p10": c10, "ms_per_step_p90": c90,
                                  "note": "eager step after an L2 flush, events around the step"}
            kept[name] = b.w
            if b is not head:
                b.free()
            if name in ALT_SCHEDULE:
                a = Bench(name, ALT_SCHEDULE[name], None, dev, rank, ws)
                a.run(K, W, R, hot=False)
                ar = a.result(peak, peak_src)
                a.free()
                res["alt_schedule"] = {k: ar[k] for k in ("schedule", "partition_size", "launches_per_step",
                                                         "ms_per_step", "ms_per_step_p10", "ms_per_step_p90",
                                                         "value", "kernel", "kernel_ms", "roofline",
                                                         "device_error_flags")}
                res["device_error_flags"] |= ar["device_error_flags"]
            per_config[name] = res
    head.free()
    clocks = sampler.stop() if not args.quick else None

    # the oracle on this host's cores (after every GPU measurement)
    cb = None
    if do_cpu:
        head_w = head.w
        if do_configs:
            for name in CONFIG_ORDER:
                w = kept[name]
                per_config[name]["cpu_baseline"] = cpu_baselines(w, per_config[name]["schedule"], args.cpu_seconds)
                if w is head_w or per_config[name]["workload"] == head_res["workload"]:
                    cb = per_config[name]["cpu_baseline"]
        if cb is None:
            cb = cpu_baselines(head_w, head.schedule, args.cpu_seconds)
        cb = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "single_thread")}

    flags = head_res["device_error_flags"] | sum(r["device_error_flags"] for r in per_config.values())
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return 0 if flags == 0 else 3
    w = head.w
    roof = dict(head_res["roofline"])
    roof["kernel"] = head_res["kernel"]
    roof["kernel_ms"] = head_res["kernel_ms"]
    roof["frac_of_nominal_8000"] = roof["achieved"] / 8000.0
    config = {"workload": w.name, "batch": w.num_seqs, "q_len": w.q_len, "heads": w.num_heads,
              "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "cache": w.cache, "schedule": head.schedule,
              "partition_size": head.partition_size, "sum_context": int(w.context_lens.sum()),
              "bytes_per_step": head.total_b, "parallelism": f"replicas x{ws}", "l2": head.l2_note(),
              "repeats": R, "headline": "the Llama-3-8B-like batched decode step: the metric names no "
                                        "workload; per_config holds all five"}
    if head.schedule == "cascade":
        config["cascade_items"] = int(head.plan[0].shape[0])
        config["plain_attention_bytes"] = step_bytes(w)[0]
    if head.schedule == "sparse":
        config["pages_listed"] = int(w.page_counts.sum())
        config["dense_attention_bytes"] = step_bytes(w)[0]
    line = {
        "metric": METRIC, "value": head_res["value"], "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": head_res["ms_per_step"], "ms_per_step_p10": head_res["ms_per_step_p10"],
        "ms_per_step_p90": head_res["ms_per_step_p90"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "steps_per_s": head_res["steps_per_s"], "tokens_per_s": head_res["tokens_per_s"],
        "roofline": roof, "hot_l2": head_res.get("hot_l2"), "cpu_baseline": cb, "e2e": e2e,
        "gpu_launches": K * head.launches, "clocks": clocks, "device_error_flags": flags,
        "per_config": per_config or None,
    }
    print(json.dumps(line))
    return 0 if flags == 0 else 3


if __name__ == "__main__":
    sys.exit(main())
