"""Host policy of sparse page-indirection decode (no GPU): it is used when the
page lists leave out at least min_sparsity of all pages [mlxcel manual "KV
Cache", §"Paged Decode Storage and Kernels": a minimum sparsity gates it]."""
import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()


def test_threshold():
    ctx = torch.tensor([160, 320], dtype=torch.int32)          # 10 + 20 pages
    counts = torch.tensor([4, 8], dtype=torch.int32)           # 12 of 30 listed: sparsity 0.6
    assert ops.pkv_sparse_worthwhile(counts, ctx, 0.6)
    assert ops.pkv_sparse_worthwhile(counts, ctx, 0.5)
    assert not ops.pkv_sparse_worthwhile(counts, ctx, 0.61)


def test_counts_clamped_and_empty():
    ctx = torch.tensor([16, 0], dtype=torch.int32)
    assert not ops.pkv_sparse_worthwhile(torch.tensor([5, 3], dtype=torch.int32), ctx, 0.0 + 1e-6)
    assert not ops.pkv_sparse_worthwhile(torch.tensor([0, 0], dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                                         0.0)


def test_bench_workload_is_sparse_enough():
    w = W.sparse_b4_32k()
    assert ops.pkv_sparse_worthwhile(w.page_counts, w.context_lens, 0.7)
    assert not ops.pkv_sparse_worthwhile(w.page_counts, w.context_lens, 0.8)
