"""Pins for the oracle's sparse page-indirection decode [mlxcel manual "KV
Cache", §"Paged Decode Storage and Kernels": sparse page-indirection decode].
Reading: each sequence lists logical pages (16-token blocks) and attends only
their stored tokens.  The oracle is pinned against torch SDPA in fp64 over K/V
gathered by torch indexing with a mask built from the lists, against its own
dense path (every page listed: bit-identical), and against closed forms (no
page: zeros; one listed token: V exactly)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_decode_attention_cache_gb300 import workloads as W
from tests.helpers import ODT, OCACHE, bits, np_i32, oracle_attention, oracle_cache_after_step


def sparse_oracle(w, cs, page_lists, page_counts, threads=4):
    return oracle.paged_attention(bits(w.q), ODT[w.src_dtype], w.scale, OCACHE[w.cache], cs["k"], cs["v"],
                                  np_i32(w.block_tables), np_i32(w.context_lens), q_len=w.q_len,
                                  threads=threads, page_lists=page_lists, page_counts=page_counts)


def used_pages(lst, cnt, ctx):
    """The pages a list selects: in order, each inside the context's pages and
    above the last one taken."""
    npages, last, out = -(-ctx // 16), -1, []
    for p in lst[:cnt]:
        if 0 <= p < npages and p > last:
            out.append(int(p))
            last = p
    return out


def sdpa_sparse(w, cs, page_lists, page_counts):
    conv = oracle.f16_bits_to_f64 if w.cache == "f16" else oracle.bf16_bits_to_f64
    k64 = torch.from_numpy(conv(cs["k"])).reshape(-1, w.num_kv_heads, w.head_dim)
    v64 = torch.from_numpy(conv(cs["v"])).reshape(-1, w.num_kv_heads, w.head_dim)
    q64 = torch.from_numpy(conv(bits(w.q)))
    g = w.num_heads // w.num_kv_heads
    table = w.block_tables.cpu().long()
    out = torch.zeros_like(q64)
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        pages = used_pages(list(page_lists[s]), int(page_counts[s]), c)
        t = torch.tensor([p * 16 + o for p in pages for o in range(16) if p * 16 + o < c], dtype=torch.long)
        if t.numel() == 0:
            continue
        slots = table[s][t // 16] * 16 + t % 16
        K = k64[slots].repeat_interleave(g, 1).transpose(0, 1)
        V = v64[slots].repeat_interleave(g, 1).transpose(0, 1)
        Q = q64[s:s + 1].transpose(0, 1)
        out[s:s + 1] = F.scaled_dot_product_attention(Q, K, V, scale=w.scale).transpose(0, 1)
    return out.numpy()


def random_lists(rng, ctx, max_pages, frac):
    B = len(ctx)
    pl = np.full((B, max_pages), -1, np.int32)
    pc = np.zeros(B, np.int32)
    for s, c in enumerate(ctx):
        n = -(-c // 16)
        sel = sorted(rng.choice(n, size=max(0, min(n, int(round(frac * n)))), replace=False).tolist()) if n else []
        pl[s, :len(sel)] = sel
        pc[s] = len(sel)
    return pl, pc


CASES = [
    # (ctx, H, Hkv, D, dtype, fraction of pages)
    ([1, 15, 16, 17, 40, 100], 4, 2, 64, "f16", 0.5),
    ([33, 7, 64, 200], 8, 2, 128, "bf16", 0.3),
    ([300, 48, 129], 8, 8, 64, "bf16", 0.8),
    ([500, 77], 16, 2, 128, "f16", 0.1),
]


@pytest.mark.parametrize("ctx,H,Hkv,D,dt,frac", CASES)
def test_sparse_matches_sdpa_over_listed_pages(ctx, H, Hkv, D, dt, frac):
    w = W.build(name="t", seed=31, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D, cache=dt)
    cs = oracle_cache_after_step(w)
    pl, pc = random_lists(np.random.default_rng(5), ctx, w.max_blocks, frac)
    got = sparse_oracle(w, cs, pl, pc)
    ref = sdpa_sparse(w, cs, pl, pc)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_every_page_listed_is_dense_bit_identical():
    ctx = [1, 16, 17, 90, 300]
    w = W.build(name="t", seed=32, context_lens=ctx, num_heads=8, num_kv_heads=2, head_dim=64, cache="bf16")
    cs = oracle_cache_after_step(w)
    pl = np.full((len(ctx), w.max_blocks), -1, np.int32)
    pc = np.zeros(len(ctx), np.int32)
    for s, c in enumerate(ctx):
        n = -(-c // 16)
        pl[s, :n] = np.arange(n)
        pc[s] = n
    got = sparse_oracle(w, cs, pl, pc)
    dense = oracle_attention(w, cs)
    assert np.array_equal(got, dense)


def test_bad_entries_are_skipped():
    """Out-of-range, repeated and decreasing entries are skipped: the result is
    that of the clean list, and SDPA over the pages a plain reading keeps."""
    ctx = [100, 64, 40]
    w = W.build(name="t", seed=33, context_lens=ctx, num_heads=4, num_kv_heads=2, head_dim=64, cache="f16")
    cs = oracle_cache_after_step(w)
    pl = np.array([[0, 3, 3, 2, 6, 7, 99, -1], [5, 1, 2, 4, 0, 0, 0, 0], [-2, 0, 2, 1, 9, 0, 0, 0]], np.int32)
    pc = np.array([8, 4, 5], np.int32)
    clean = np.array([[0, 3, 6, -1], [1, 2, -1, -1], [0, 2, -1, -1]], np.int32)
    cc = np.array([3, 2, 2], np.int32)
    got = sparse_oracle(w, cs, pl, pc)
    want = sparse_oracle(w, cs, clean, cc)
    assert np.array_equal(got, want)
    np.testing.assert_allclose(got, sdpa_sparse(w, cs, clean, cc), rtol=1e-12, atol=1e-13)


def test_no_page_gives_zeros_and_one_token_gives_v():
    ctx = [33, 20]
    w = W.build(name="t", seed=34, context_lens=ctx, num_heads=4, num_kv_heads=2, head_dim=64, cache="bf16")
    cs = oracle_cache_after_step(w)
    pl = np.array([[2, -1], [0, -1]], np.int32)   # seq 0: page 2 holds only token 32
    pc = np.array([1, 0], np.int32)
    got = sparse_oracle(w, cs, pl, pc)
    assert np.array_equal(got[1], np.zeros_like(got[1]))
    pb = int(w.block_tables[0, 2])
    v = oracle.bf16_bits_to_f64(cs["v"])[pb, 0]                        # token 32 = slot 0 of page 2
    for h in range(4):
        assert np.array_equal(got[0, h], v[h // 2])
