"""The algorithmic-bytes accounting behind bench.py's roofline, checked by direct
counts on small cases: dense decode counts every visible (token, kv head) K and
V row once; cascade counts a shared prefix once per item; sparse counts only the
listed pages' stored tokens."""
import pytest

from paged_decode_attention_cache_gb300 import bytes_model as BM


def kv_row(cache, D=128):
    kb, vb = BM.row_bytes(cache, D)
    return kb + vb


@pytest.mark.parametrize("cache", ["bf16", "k8v4"])
def test_dense_counts_every_visible_row_once(cache):
    ctx = [1, 16, 17, 300]
    H, Hkv, D = 32, 8, 128
    got = BM.attention_bytes(ctx, 1, H, Hkv, D, cache)
    kv = sum(ctx) * Hkv * kv_row(cache, D)
    qo = len(ctx) * H * D * 4
    tables = 4 * sum(-(-c // 16) for c in ctx) + 4 * len(ctx)
    assert got == kv + qo + tables


def test_window_counts_only_the_last_tokens():
    ctx, W = [100, 4096, 30], 64
    got = BM.attention_bytes(ctx, 1, 32, 8, 128, "bf16", sliding_window=W)
    full = BM.attention_bytes([min(c, W) for c in ctx], 1, 32, 8, 128, "bf16")
    # same rows; the window may start inside a block, so its table entries differ by at most one per sequence
    assert abs(got - full) <= 4 * len(ctx)


def test_cascade_without_items_is_dense_kv():
    ctx = [200, 333, 64]
    dense = BM.attention_bytes(ctx, 1, 32, 8, 128, "bf16")
    assert BM.cascade_attention_bytes(ctx, [], [], 32, 8, 128, "bf16") == dense


def test_cascade_reads_a_shared_prefix_once():
    ctx = [200, 333, 64, 500]
    members, blocks = [[0, 1, 3, -1]], [4]          # three members share 4 pages (64 tokens)
    got = BM.cascade_attention_bytes(ctx, members, blocks, 32, 8, 128, "bf16")
    dense = BM.attention_bytes(ctx, 1, 32, 8, 128, "bf16")
    saved_rows = (3 - 1) * 4 * 16                   # two extra copies of the prefix are not read
    saved_tables = (3 - 1) * 4 * 4
    assert dense - got == saved_rows * 8 * kv_row("bf16") + saved_tables


def test_sparse_every_page_is_dense_kv():
    ctx = [17, 100, 512]
    lists = [list(range(-(-c // 16))) for c in ctx]
    counts = [len(x) for x in lists]
    got = BM.sparse_attention_bytes(ctx, lists, counts, 32, 8, 128, "bf16")
    dense_kv = sum(ctx) * 8 * kv_row("bf16")
    overhead = 4 * sum(counts) + 12 * sum(counts) + 12 * len(ctx)
    assert got == dense_kv + len(ctx) * 32 * 128 * 4 + overhead


def test_sparse_counts_listed_pages_and_the_tail():
    ctx = [40]                                       # pages 0, 1 full, page 2 holds 8 tokens
    for lst, tokens in (([0], 16), ([2], 8), ([0, 2], 24), ([2, 0], 8), ([1, 1, 5], 16)):
        got = BM.sparse_attention_bytes(ctx, [lst], [len(lst)], 4, 2, 64, "f16")
        pages = {0: 0, 16: 1, 8: 1, 24: 2}[tokens] if lst != [1, 1, 5] else 1
        want = tokens * 2 * (2 * 64 * 2) + 4 * 64 * 4 + 4 * len(lst) + 12 * pages + 12
        assert got == want, (lst, got, want)
