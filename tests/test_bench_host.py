"""Host-side pieces of bench.py that need no GPU: the repeat statistics, the
byte counts of a sample of sequences, and the oracle baseline on a small
workload (single-thread and all-core legs)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_decode_attention_cache_gb300 import bytes_model as BM, workloads as W  # noqa: E402


def test_summary_median_and_percentiles():
    med, p10, p90 = bench.summary([5.0, 1.0, 3.0, 2.0, 4.0])
    assert med == 3.0
    assert p10 == pytest.approx(1.4) and p90 == pytest.approx(4.6)
    assert bench.summary([2.5]) == (2.5, 2.5, 2.5)


def test_sample_bytes_add_up_to_the_whole_batch():
    w = W.build(name="t", seed=3, context_lens=[17, 300, 64, 1], num_heads=8, num_kv_heads=2, head_dim=64,
                cache="bf16")
    whole, wr = bench.step_bytes(w)
    parts = sum(bench.step_bytes(w, seqs=[s])[0] for s in range(4))
    # the per-sequence counts add up (every term is per sequence)
    assert parts == whole
    assert wr == BM.write_bytes(int(w.slot_new.numel()), 2, 64, "bf16")


def test_cpu_baseline_single_and_all_core():
    w = W.build(name="t", seed=4, context_lens=[40, 90, 200], num_heads=8, num_kv_heads=2, head_dim=64,
                cache="f16")
    cb = bench.cpu_baselines(w, "fused", 0.05)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] == (os.cpu_count() or 1)
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert "sequences" in cb["sample"]
    split = bench.cpu_baseline(W.build(name="t", seed=5, context_lens=[600], num_heads=4, num_kv_heads=2,
                                       head_dim=64, cache="bf16", partition_size=128), "split", 1, 0.05)
    assert "LSE reduce" in split["sample"]
