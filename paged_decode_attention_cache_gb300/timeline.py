"""Where a launch's time goes: a %globaltimer timeline of back-to-back steps.

    python -m paged_decode_attention_cache_gb300.timeline --workload llama3_8b_batch8

Builds libpkv_timeline.so (the same sources with -DPKV_TIMELINE: thread 0 of
every CTA stamps fixed points of its run, see attention_impl.cuh), steps the
bench's workload in one CUDA graph of back-to-back launches over its rotating
input replicas, and prints markdown tables of each phase's time after the
previous launch's last CTA ended (the restart gap, the stream, the tail) and of
each lane range.  The stamps themselves cost time; the launch period it prints
is that of the instrumented library, not a bench value.
"""
from __future__ import annotations

import argparse
import ctypes
import sys

import numpy as np
import torch

from . import build, ops

LAUNCHES, CTAS, WORDS, SEGS = 64, 160, 32, 6   # kTlLaunches, kTlCtas, kTlWords, kTlSegs


def record(workload: str, steps: int):
    ops.select_library(build.build(timeline=True))
    L = ops.lib()
    L.pkv_timeline_attach.restype = None
    L.pkv_timeline_attach.argtypes = [ctypes.c_void_p]
    import bench   # the repository root is on sys.path under `python -m`
    torch.cuda.set_device(0)
    b = bench.Bench(workload, None, None, "cuda:0", 0, 1)
    buf = torch.zeros(1 + LAUNCHES * CTAS * WORDS, dtype=torch.int64, device="cuda")
    L.pkv_timeline_attach(buf.data_ptr())
    for i in range(max(3, b.reps)):
        b.steps[i % b.reps].step()
    graphs = bench.capture_steps(lambda k: b.steps[k % b.reps].step(), steps)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    buf.zero_()
    torch.cuda.synchronize()
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    flags = b.flags if hasattr(b, "flags") else 0
    for s in b.steps:
        flags |= s.error_flags()
    t = buf.cpu().numpy()
    n_entries = int(t[0])
    rec = t[1:].reshape(LAUNCHES, CTAS, WORDS).astype(np.int64)
    return b, rec, n_entries, flags


def analyse(rec: np.ndarray, n_launches: int, hkv: int):
    grid = int((rec[0, :, 0] > 0).sum())
    rec = rec[:n_launches, :grid]
    nseg = (rec[:, :, 28] & 0xff).astype(int)
    seg_t = rec[:, :, 4:4 + 4 * SEGS].reshape(n_launches, grid, SEGS, 4)
    last = np.clip(nseg - 1, 0, SEGS - 1)
    idx_l, idx_c = np.meshgrid(np.arange(n_launches), np.arange(grid), indexing="ij")
    end = np.where(nseg > 0, seg_t[idx_l, idx_c, last, 3], 0)
    merged = np.where(nseg > 0, seg_t[idx_l, idx_c, last, 1], 0)
    comb_end = ((rec[:, :, 28] >> (8 + last)) & 1).astype(bool) & (nseg > 0)
    blocks = np.zeros((n_launches, grid), dtype=int)
    for k in range(4):
        blocks += np.where(k < nseg, (rec[:, :, 29] >> (16 * k)) & 0xffff, 0).astype(int)
    rows, periods = [], []
    for l in range(2, n_launches):
        prev_end = end[l - 1][end[l - 1] > 0].max()
        periods.append((end[l][end[l] > 0].max() - prev_end) / 1e3)
        rel = lambda x: np.where(x > 0, (x - prev_end) / 1e3, np.nan)
        rows.append(np.stack([rel(rec[l, :, 0]), rel(rec[l, :, 1]), rel(rec[l, :, 2]), rel(rec[l, :, 3]),
                              rel(merged[l]), rel(end[l])], axis=-1))
    R = np.stack(rows)   # [launch, cta, phase]
    # the last segment's end phases: merged -> published (pieces only) -> end
    pub = np.where(nseg > 0, seg_t[idx_l, idx_c, last, 2], 0)
    piece_end = ((rec[:, :, 28] >> (16 + last)) & 1).astype(bool) & (nseg > 0)
    tails = {"merged_to_published": np.where(piece_end & (pub > 0), (pub - merged) / 1e3, np.nan)[2:],
             "published_to_end": np.where(piece_end & (pub > 0), (end - pub) / 1e3, np.nan)[2:],
             "merged_to_end": np.where(nseg > 0, (end - merged) / 1e3, np.nan)[2:],
             "piece": piece_end[2:]}
    return grid, R, np.array(periods), nseg[2:], blocks[2:], comb_end[2:], tails


def report(workload, b, grid, R, periods, nseg, blocks, comb_end, hkv, flags, tails=None):
    out = []
    out.append(f"{workload} ({b.schedule}), grid {grid} = {grid // hkv} lane ranges x {hkv} kv heads; "
               f"{len(periods)} launches; device error flags {flags:#x}\n")
    out.append(f"Launch period (last CTA end to last CTA end), instrumented: median {np.median(periods):.2f} us\n")
    out.append("| phase (us after the previous launch's last CTA end) | p10 | median | max |")
    out.append("|---|---|---|---|")
    names = ["CTA entry", "plan done", "first copies issued (after the grid dependency wait)",
             "first block in shared memory", "last segment's blocks merged", "CTA end"]
    for i, n in enumerate(names):
        x = R[:, :, i]
        x = x[np.isfinite(x)]
        out.append(f"| {n} | {np.percentile(x, 10):.2f} | {np.median(x):.2f} | {x.max():.2f} |")
    out.append("")
    if tails is not None:
        out.append("| a CTA's last segment (µs, median) | CTAs | merged → published | published → end | merged → end |")
        out.append("|---|---|---|---|---|")
        kinds = (("whole (sequence, kv head) pair", ~tails["piece"]),
                 ("piece, not the last of its pair", tails["piece"] & ~comb_end),
                 ("piece that combines its pair", tails["piece"] & comb_end))
        for name, sel in kinds:
            if not sel.any():
                continue
            med = lambda a: f"{np.nanmedian(a[sel]):.2f}" if np.isfinite(a[sel]).any() else "–"
            out.append(f"| {name} | {sel.sum() / len(sel):.0f} | {med(tails['merged_to_published'])} | "
                       f"{med(tails['published_to_end'])} | {med(tails['merged_to_end'])} |")
        out.append("")
    out.append("| lane range | segments | blocks | combines at its end | first copies | last blocks merged | end |")
    out.append("|---|---|---|---|---|---|---|")
    nl = grid // hkv
    for r in range(nl):
        cols = [r * hkv + h for h in range(hkv)]
        sel = lambda a: a[:, cols]
        out.append(f"| {r} | {np.median(sel(nseg)):.0f} | {np.median(sel(blocks)):.0f} | "
                   f"{sel(comb_end).mean():.2f} | {np.nanmedian(sel(R[:, :, 2])):.2f} | "
                   f"{np.nanmedian(sel(R[:, :, 4])):.2f} | {np.nanmedian(sel(R[:, :, 5])):.2f} |")
    return "\n".join(out)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--workload", default="llama3_8b_batch8")
    ap.add_argument("--steps", type=int, default=LAUNCHES, help=f"launches recorded (at most {LAUNCHES})")
    a = ap.parse_args(argv)
    steps = min(a.steps, LAUNCHES)
    b, rec, n_entries, flags = record(a.workload, steps)
    hkv = b.w.num_kv_heads
    grid, R, periods, nseg, blocks, comb_end, tails = analyse(rec, steps, hkv)
    print(report(a.workload, b, grid, R, periods, nseg, blocks, comb_end, hkv, flags, tails))
    return 0


if __name__ == "__main__":
    sys.exit(main())
