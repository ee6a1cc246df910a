"""Pins for the oracle's attention, split-KV partials and LSE reduce.

Each pin fixes the oracle against something other than itself: a library
routine (torch SDPA in fp64 over K/V gathered by torch indexing), closed forms
(one visible token returns V; identical keys return mean V), the paging
invariants the pages state (an identity table is a contiguous cache; physical
block ids are arbitrary), GQA as repeated kv heads, causal verify rows as
shorter single-query decodes, and a hand-worked LSE combination.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_decode_attention_cache_gb300 import workloads as W
from tests.helpers import bits, np_i32, oracle_attention, oracle_cache_after_step


def _pool64(w, cs, which):
    conv = oracle.f16_bits_to_f64 if w.cache == "f16" else oracle.bf16_bits_to_f64
    return torch.from_numpy(conv(cs[which]))


def sdpa_reference(w, cs):
    """torch SDPA (fp64, CPU) over K/V gathered with torch indexing."""
    k64, v64 = _pool64(w, cs, "k"), _pool64(w, cs, "v")
    conv = oracle.f16_bits_to_f64 if w.src_dtype == "f16" else oracle.bf16_bits_to_f64
    q64 = torch.from_numpy(conv(bits(w.q)))
    g = w.num_heads // w.num_kv_heads
    table = w.block_tables.cpu().long()
    out = torch.zeros_like(q64)
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        if c == 0:
            continue
        t = torch.arange(c)
        slots = table[s][t // 16] * 16 + t % 16
        K = k64.reshape(-1, w.num_kv_heads, w.head_dim)[slots].repeat_interleave(g, 1).transpose(0, 1)
        V = v64.reshape(-1, w.num_kv_heads, w.head_dim)[slots].repeat_interleave(g, 1).transpose(0, 1)
        Q = q64[s * w.q_len:(s + 1) * w.q_len].transpose(0, 1)          # [H, q_len, D]
        j = torch.arange(w.q_len)[:, None]
        mask = t[None, :] < (c - w.q_len + j + 1)                        # [q_len, c]
        if w.sliding_window > 0:                                         # last W stored tokens
            mask = mask & (t[None, :] >= c - w.sliding_window)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=w.scale)
        empty = ~mask.any(1)
        o[:, empty] = 0.0
        out[s * w.q_len:(s + 1) * w.q_len] = o.transpose(0, 1)
    return out.numpy()


CASES = [
    # (ctx list, H, Hkv, D, q_len, dtype)
    ([1, 15, 16, 17, 40], 4, 2, 64, 1, "f16"),
    ([33, 7, 64], 8, 2, 128, 1, "bf16"),
    ([20, 48], 4, 4, 64, 1, "bf16"),
    ([5, 31, 16], 8, 1, 64, 1, "f16"),
    ([9, 40, 4], 8, 2, 64, 3, "bf16"),
    ([64, 17], 8, 8, 128, 2, "f16"),
]


@pytest.mark.parametrize("ctx,H,Hkv,D,ql,dt", CASES)
def test_oracle_matches_sdpa(ctx, H, Hkv, D, ql, dt):
    w = W.build(name="t", seed=11, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=dt, q_len=ql)
    cs = oracle_cache_after_step(w)
    got = oracle_attention(w, cs)
    ref = sdpa_reference(w, cs)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_single_token_returns_v_exactly():
    w = W.build(name="t", seed=3, context_lens=[1, 1, 1], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16")
    cs = oracle_cache_after_step(w)
    got = oracle_attention(w, cs)
    v = oracle.bf16_bits_to_f64(cs["v"]).reshape(-1, 2, 64)
    for s in range(3):
        slot = int(w.block_tables[s, 0]) * 16
        for h in range(4):
            assert np.array_equal(got[s, h], v[slot, h // 2])


def test_uniform_keys_give_mean_v():
    w = W.build(name="t", seed=4, context_lens=[37], num_heads=4, num_kv_heads=1, head_dim=64,
                cache="f16", new_tokens="none")
    cs = oracle_cache_after_step(w)
    k = cs["k"].reshape(-1, 1, 64)
    t = np.arange(37)
    slots = np_i32(w.block_tables)[0][t // 16] * 16 + t % 16
    k[slots] = k[slots[0]]                      # every visible key identical
    got = oracle_attention(w, cs)
    v = oracle.f16_bits_to_f64(cs["v"]).reshape(-1, 1, 64)[slots, 0]
    for h in range(4):
        np.testing.assert_allclose(got[0, h], v.mean(0), rtol=0, atol=1e-14)


def test_identity_table_equals_contiguous_cache():
    """With an identity block table the paged cache is a contiguous cache."""
    w = W.build(name="t", seed=5, context_lens=[70], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16", identity_table=True, new_tokens="none", num_blocks=5)
    cs = oracle_cache_after_step(w)
    got = oracle_attention(w, cs)
    k = torch.from_numpy(oracle.bf16_bits_to_f64(cs["k"]).reshape(-1, 2, 64)[:70])
    v = torch.from_numpy(oracle.bf16_bits_to_f64(cs["v"]).reshape(-1, 2, 64)[:70])
    q = torch.from_numpy(oracle.bf16_bits_to_f64(bits(w.q)))[0]         # [H, D]
    K = k.repeat_interleave(2, 1).transpose(0, 1)
    V = v.repeat_interleave(2, 1).transpose(0, 1)
    ref = F.scaled_dot_product_attention(q[:, None], K, V, scale=w.scale)[:, 0]
    np.testing.assert_allclose(got[0], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_physical_block_permutation_invariance():
    w = W.build(name="t", seed=6, context_lens=[50, 23], num_heads=8, num_kv_heads=2, head_dim=64,
                cache="f16", num_blocks=12, new_tokens="none")
    cs = oracle_cache_after_step(w)
    base = oracle_attention(w, cs)
    perm = np.random.default_rng(0).permutation(12)        # new id of physical block b
    k2 = np.empty_like(cs["k"])
    v2 = np.empty_like(cs["v"])
    k2[perm] = cs["k"]
    v2[perm] = cs["v"]
    table = np_i32(w.block_tables)
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    w.block_tables = torch.from_numpy(table2)
    got = oracle_attention(w, {"k": k2, "v": v2})
    assert np.array_equal(got, base)


@pytest.mark.parametrize("P", [16, 32, 80, 512])
def test_split_partials_and_reduce_equal_single_pass(P):
    w = W.build(name="t", seed=7, context_lens=[1, 95, 160, 17], num_heads=4, num_kv_heads=2,
                head_dim=64, cache="bf16", q_len=2)
    cs = oracle_cache_after_step(w)
    single = oracle_attention(w, cs)
    NP = -(-w.max_blocks * 16 // P)
    _, (po, pm, pl) = oracle_attention(w, cs, partition_size=P, max_partitions=NP)
    red = oracle.lse_reduce(po, pm, pl)
    np.testing.assert_allclose(red, single, rtol=1e-12, atol=1e-14)
    # each partial is attention over exactly its partition's visible tokens
    for r in range(w.num_rows):
        s, j = divmod(r, w.q_len)
        vis = max(0, int(w.context_lens[s]) - w.q_len + j + 1)
        for p in range(NP):
            n = max(0, min(vis, (p + 1) * P) - p * P)
            assert (pl[r, :, p] > 0).all() == (n > 0)
            if n == 0:
                assert np.isneginf(pm[r, :, p]).all() and not po[r, :, p].any()
            else:
                assert (pl[r, :, p] >= 1.0).all() and (pl[r, :, p] <= n * (1 + 1e-12)).all()


def test_gqa_equals_mha_with_repeated_kv_heads():
    w = W.build(name="t", seed=8, context_lens=[29, 64], num_heads=8, num_kv_heads=2, head_dim=64,
                cache="f16")
    cs = oracle_cache_after_step(w)
    gqa = oracle_attention(w, cs)
    rep = {"k": np.repeat(cs["k"], 4, axis=2).copy(), "v": np.repeat(cs["v"], 4, axis=2).copy()}
    w.num_kv_heads = 8
    mha = oracle_attention(w, rep)
    assert np.array_equal(gqa, mha)


def test_verify_rows_equal_shorter_single_query_decodes():
    w = W.build(name="t", seed=9, context_lens=[40, 21], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16", q_len=4)
    cs = oracle_cache_after_step(w)
    ver = oracle_attention(w, cs)
    for s in range(2):
        for j in range(4):
            r = s * 4 + j
            c = int(w.context_lens[s]) - 4 + j + 1
            one = oracle.paged_attention(bits(w.q)[r:r + 1], oracle.BF16, w.scale,
                                         oracle.CACHE_BF16, cs["k"], cs["v"],
                                         np_i32(w.block_tables)[s:s + 1],
                                         np.array([c], np.int32), q_len=1)
            assert np.array_equal(one[0], ver[r])


def test_empty_context_gives_zeros():
    w = W.build(name="t", seed=10, context_lens=[0, 3], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16", q_len=4, new_tokens="none", max_blocks=1)
    got = oracle_attention(w)
    assert not got[0:4].any()                 # no visible token at all
    assert not got[4:5].any()                 # ctx 3 with 4 drafts: draft 0 sees nothing
    assert np.isfinite(got).all() and got[5:8].any()


def test_lse_reduce_worked_example():
    # partition 0: m = 0, l = 1, o = 1;  partition 1: m = ln 3, l = 1, o = 0
    # weights 1/3 and 1 -> out = (1/3) / (4/3) = 1/4; partition 2 empty is ignored
    po = np.array([[[[1.0], [0.0], [0.0]]]])
    pm = np.array([[[0.0, math.log(3.0), -np.inf]]])
    pl = np.array([[[1.0, 1.0, 0.0]]])
    out = oracle.lse_reduce(po, pm, pl)
    assert abs(out[0, 0, 0] - 0.25) < 1e-15
    assert not oracle.lse_reduce(po, np.full_like(pm, -np.inf), np.zeros_like(pl)).any()


def test_oracle_rejects_out_of_range_block():
    w = W.build(name="t", seed=12, context_lens=[20], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16", new_tokens="none")
    cs = oracle_cache_after_step(w)
    w.block_tables = w.block_tables.clone()
    w.block_tables[0, 1] = w.num_blocks
    with pytest.raises(ValueError):
        oracle_attention(w, cs)


def test_nan_sentinel_reaches_output_when_read():
    """The NaN fill of unused slots is live: a context one token too long (its
    slot never written) makes the output NaN."""
    w = W.build(name="t", seed=13, context_lens=[20], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16", new_tokens="none", max_blocks=2)
    cs = oracle_cache_after_step(w)
    w.context_lens = torch.tensor([21], dtype=torch.int32)
    assert np.isnan(oracle_attention(w, cs)).all()


# ---------------------------------------------------------------- sliding window
# [MTPLX-2 §"Sliding-Window Memory Control": the visible part of the cache is
#  trimmed to the last `window` stored tokens; older ones are masked.]

WINDOW_CASES = [
    # (ctx list, H, Hkv, D, q_len, dtype, window)
    ([1, 15, 16, 17, 40, 100], 4, 2, 64, 1, "f16", 16),
    ([33, 7, 64, 200], 8, 2, 128, 1, "bf16", 17),
    ([9, 40, 4, 70], 8, 2, 64, 3, "bf16", 20),
    ([64, 17, 130], 8, 8, 128, 2, "f16", 5),
    ([50, 3], 4, 4, 64, 1, "bf16", 1),
]


@pytest.mark.parametrize("ctx,H,Hkv,D,ql,dt,win", WINDOW_CASES)
def test_window_matches_sdpa_over_the_last_tokens(ctx, H, Hkv, D, ql, dt, win):
    w = W.build(name="t", seed=21, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=dt, q_len=ql, sliding_window=win)
    cs = oracle_cache_after_step(w)
    got = oracle_attention(w, cs)
    ref = sdpa_reference(w, cs)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_window_at_least_the_context_changes_nothing():
    kw = dict(name="t", seed=22, context_lens=[1, 31, 64, 97], num_heads=8, num_kv_heads=2,
              head_dim=64, cache="bf16", q_len=2)
    w0 = W.build(**kw)
    cs = oracle_cache_after_step(w0)
    base = oracle_attention(w0, cs)
    for win in (97, 98, 4096):
        w = W.build(**kw, sliding_window=win)
        assert np.array_equal(oracle_attention(w, cs), base)


def test_window_of_one_token_returns_its_v():
    w = W.build(name="t", seed=23, context_lens=[5, 40, 1], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="bf16", sliding_window=1)
    cs = oracle_cache_after_step(w)
    got = oracle_attention(w, cs)
    v = oracle.bf16_bits_to_f64(cs["v"]).reshape(-1, 2, 64)
    table = np_i32(w.block_tables)
    for s in range(w.num_seqs):
        t = int(w.context_lens[s]) - 1
        slot = int(table[s, t // 16]) * 16 + t % 16
        for h in range(4):
            assert np.array_equal(got[s, h], v[slot, h // 2])


def test_window_equals_shorter_table_of_the_last_tokens():
    # dropping the first ctx-W tokens (whole blocks) from the table leaves the
    # same visible set when ctx-W is a multiple of 16
    w = W.build(name="t", seed=24, context_lens=[80, 48], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="f16", sliding_window=32)
    cs = oracle_cache_after_step(w)
    got = oracle_attention(w, cs)
    table = np_i32(w.block_tables)
    short = np.full_like(table, -1)
    short[0, :2] = table[0, 3:5]
    short[1, :2] = table[1, 1:3]
    conv = oracle.f16_bits_to_f64
    ref = oracle.paged_attention(bits(w.q), oracle.F16, w.scale, oracle.CACHE_F16, cs["k"], cs["v"],
                                 short, np.array([32, 32], np.int32))
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("P", [16, 48, 64])
def test_window_split_partials_reduce_to_single_pass(P):
    w = W.build(name="t", seed=25, context_lens=[1, 95, 160, 17, 200], num_heads=4, num_kv_heads=2,
                head_dim=64, cache="bf16", q_len=2, sliding_window=37)
    cs = oracle_cache_after_step(w)
    single = oracle_attention(w, cs)
    NP = -(-w.max_blocks * 16 // P)
    _, (po, pm, pl) = oracle_attention(w, cs, partition_size=P, max_partitions=NP)
    np.testing.assert_allclose(oracle.lse_reduce(po, pm, pl), single, rtol=1e-12, atol=1e-14)
    # partitions wholly before the window are empty
    for s in range(w.num_seqs):
        lo = max(0, int(w.context_lens[s]) - 37)
        for p in range(NP):
            if (p + 1) * P <= lo:
                rows = slice(s * 2, s * 2 + 2)
                assert np.isneginf(pm[rows, :, p]).all() and not pl[rows, :, p].any()
