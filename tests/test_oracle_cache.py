"""Pins for the oracle's cache writes, gathers, quantiser and the bytes model."""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_decode_attention_cache_gb300 import bytes_model
from paged_decode_attention_cache_gb300 import workloads as W
from tests.helpers import bits, np_i32, np_i64, oracle_attention, oracle_cache_after_step

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- reshape / gather

def test_reshape_and_cache_matches_torch_scatter_and_leaves_rest():
    rng = np.random.default_rng(0)
    NB, Hkv, D, T = 6, 2, 64, 11
    kc = rng.integers(0, 1 << 16, (NB, 16, Hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, (NB, 16, Hkv, D), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, (T, Hkv, D), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, (T, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[3] = -1                        # padding
    slots[7] = NB * 16 + 5               # out of range
    ref_k, ref_v = torch.from_numpy(kc.view(np.int16).copy()), torch.from_numpy(vc.view(np.int16).copy())
    ok = (slots >= 0) & (slots < NB * 16)
    ref_k.view(-1, Hkv, D)[torch.from_numpy(slots[ok])] = torch.from_numpy(kn.view(np.int16)[ok])
    ref_v.view(-1, Hkv, D)[torch.from_numpy(slots[ok])] = torch.from_numpy(vn.view(np.int16)[ok])
    nbad = oracle.reshape_and_cache(kc, vc, kn, vn, slots)
    assert nbad == 1
    assert np.array_equal(kc.view(np.int16), ref_k.numpy())
    assert np.array_equal(vc.view(np.int16), ref_v.numpy())


def test_gather_round_trip_and_matches_torch_indexing():
    w = W.build(name="t", seed=1, context_lens=[5, 33, 16, 0, 47], num_heads=4, num_kv_heads=2,
                head_dim=64, cache="bf16")
    cs = oracle_cache_after_step(w)
    cu = w.cu_seq_lens().numpy()
    ko, vo = oracle.gather_kv_cache(cs["k"], cs["v"], np_i32(w.block_tables),
                                    np_i32(w.context_lens), cu)
    table = w.block_tables.long()
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        t = torch.arange(c)
        slots = (table[s][t // 16] * 16 + t % 16).numpy()
        assert np.array_equal(ko[cu[s]:cu[s] + c], cs["k"].reshape(-1, 2, 64)[slots])
        assert np.array_equal(vo[cu[s]:cu[s] + c], cs["v"].reshape(-1, 2, 64)[slots])
    # the rows written by the step come back unchanged
    new_k = bits(w.k_new)
    pos = [cu[s] + int(w.context_lens[s]) - 1 for s in range(w.num_seqs) if int(w.context_lens[s])]
    assert np.array_equal(ko[pos], new_k)


def test_gather_rejects_bad_block():
    w = W.build(name="t", seed=2, context_lens=[20], num_heads=4, num_kv_heads=2, head_dim=64,
                cache="f16")
    cs = oracle_cache_after_step(w)
    bt = np_i32(w.block_tables)
    bt[0, 1] = -3
    with pytest.raises(ValueError):
        oracle.gather_kv_cache(cs["k"], cs["v"], bt, np_i32(w.context_lens), w.cu_seq_lens().numpy())


# ---------------------------------------------------------------- quantiser

def _quant_one(k_vals, v_vals, dtype="bf16"):
    """Quantise one token of one kv head (D = len(k_vals)); returns the cache."""
    D = len(k_vals)
    conv = oracle.f32_to_bf16_bits if dtype == "bf16" else oracle.f32_to_f16_bits
    kn = conv(np.asarray(k_vals, np.float32)).reshape(1, 1, D)
    vn = conv(np.asarray(v_vals, np.float32)).reshape(1, 1, D)
    qc = oracle.QuantCache(1, 1, D)
    oracle.quantize_kv(qc, kn, vn, oracle.BF16 if dtype == "bf16" else oracle.F16,
                       np.array([0], np.int64))
    return qc


def _unpack_v(qc):
    lo = (qc.v_q & 0x0f).astype(np.int64)
    hi = (qc.v_q >> 4).astype(np.int64)
    return np.stack([lo, hi], -1).reshape(qc.v_q.shape[:-1] + (qc.v_q.shape[-1] * 2,))


def test_quantiser_worked_example_ties_to_even():
    D = 64
    k = np.zeros(D, np.float32)
    k[:6] = [127.0, -63.5, 0.5, 1.5, 2.5, -126.5]     # a = 127 -> scale exactly 1
    v = np.zeros(D, np.float32)
    v[:32] = np.arange(32) % 16                        # group 0: lo 0, hi 15 -> scale 1, zero 0
    v[5] = 2.5
    v[7] = 3.5
    v[32:] = 7.0                                       # group 1 constant -> scale 0, codes 0
    qc = _quant_one(k, v)
    assert qc.k_scale[0, 0, 0] == 0x3c00               # fp16 1.0
    assert list(qc.k_q[0, 0, 0, :6]) == [127, -64, 0, 2, 2, -126]
    codes = _unpack_v(qc)[0, 0, 0]
    exp0 = (np.arange(32) % 16).copy()
    exp0[5], exp0[7] = 2, 4
    assert list(codes[:32]) == list(exp0)
    assert not codes[32:].any()
    assert qc.v_scale[0, 0, 0, 0] == 0x3c00 and qc.v_zero[0, 0, 0, 0] == 0
    assert qc.v_scale[0, 0, 0, 1] == 0 and qc.v_zero[0, 0, 0, 1] == 0x4700   # fp16 7.0
    # nibble order: dim 1 (code 1) sits in the high nibble of byte 0, dim 0 (code 0) in the low
    assert qc.v_q[0, 0, 0, 0] == 0x10


def test_quantiser_error_bounds_and_code_ranges():
    w = W.build(name="t", seed=3, context_lens=[64, 80], num_heads=8, num_kv_heads=2,
                head_dim=128, cache="k8v4")
    cs = oracle_cache_after_step(w)
    qc = cs["qc"]
    # source values of every written slot, in write order
    k_src = np.concatenate([oracle.bf16_bits_to_f64(bits(w.k_hist)), oracle.bf16_bits_to_f64(bits(w.k_new))])
    v_src = np.concatenate([oracle.bf16_bits_to_f64(bits(w.v_hist)), oracle.bf16_bits_to_f64(bits(w.v_new))])
    slots = np.concatenate([np_i64(w.slot_hist), np_i64(w.slot_new)])
    blk, off = slots // 16, slots % 16
    ks = oracle.f16_bits_to_f64(qc.k_scale[blk, :, off])                 # [T, Hkv]
    kc = qc.k_q[blk, off].astype(np.float64)                             # [T, Hkv, D]
    assert (np.abs(kc) <= 127).all()
    amax = np.abs(k_src).max(-1)
    assert np.all(np.abs(ks - amax / 127) <= ks * 2.0 ** -10 + 1e-30)    # fp16 rounding of a/127
    assert np.all(np.abs(kc * ks[..., None] - k_src) <= ks[..., None] * 0.5 * (1 + 2.0 ** -9))
    vc = _unpack_v(qc)[blk, off].astype(np.float64)                      # [T, Hkv, D]
    assert ((vc >= 0) & (vc <= 15)).all()
    vs = oracle.f16_bits_to_f64(qc.v_scale[blk, :, off])                 # [T, Hkv, G]
    vz = oracle.f16_bits_to_f64(qc.v_zero[blk, :, off])
    vs_d = np.repeat(vs, 32, -1)
    vz_d = np.repeat(vz, 32, -1)
    deq = vc * vs_d + vz_d
    grp = v_src.reshape(v_src.shape[:-1] + (4, 32))
    lo, hi = grp.min(-1), grp.max(-1)
    slack = np.repeat(np.abs(vz - lo) + 16 * np.abs(vs - (hi - lo) / 15), 32, -1)
    assert np.all(np.abs(deq - v_src) <= 0.5 * vs_d + slack + 1e-12)


def test_k8v4_attention_matches_sdpa_over_independent_dequant():
    """The oracle's K8/V4 attention equals SDPA over codes unpacked and scaled by
    numpy from the documented layout (scales [NB, Hkv, 16], nibbles low-first)."""
    w = W.build(name="t", seed=4, context_lens=[40, 77, 3], num_heads=8, num_kv_heads=2,
                head_dim=64, cache="k8v4")
    cs = oracle_cache_after_step(w)
    qc = cs["qc"]
    got = oracle_attention(w, cs)
    NB = qc.num_blocks
    ks = oracle.f16_bits_to_f64(qc.k_scale).transpose(0, 2, 1)            # [NB, 16, Hkv]
    k64 = qc.k_q.astype(np.float64) * ks[..., None]
    vs = np.repeat(oracle.f16_bits_to_f64(qc.v_scale).transpose(0, 2, 1, 3), 32, -1)
    vz = np.repeat(oracle.f16_bits_to_f64(qc.v_zero).transpose(0, 2, 1, 3), 32, -1)
    v64 = _unpack_v(qc) * vs + vz
    q64 = torch.from_numpy(oracle.bf16_bits_to_f64(bits(w.q)))
    table = w.block_tables.long()
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        t = torch.arange(c)
        slots = (table[s][t // 16] * 16 + t % 16).numpy()
        K = torch.from_numpy(k64.reshape(NB * 16, 2, 64)[slots]).repeat_interleave(4, 1).transpose(0, 1)
        V = torch.from_numpy(v64.reshape(NB * 16, 2, 64)[slots]).repeat_interleave(4, 1).transpose(0, 1)
        ref = F.scaled_dot_product_attention(q64[s][:, None], K, V, scale=w.scale)[:, 0]
        np.testing.assert_allclose(got[s], ref.numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- dequantising gather

@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_dequant_gather_matches_numpy_torch_rounding(out):
    """Codes unpacked and scaled by numpy from the documented layout, gathered
    by numpy indexing, rounded fp64 -> fp32 -> out dtype by torch (RNE)."""
    w = W.build(name="t", seed=9, context_lens=[40, 77, 3, 16], num_heads=8, num_kv_heads=2,
                head_dim=64, cache="k8v4")
    cs = oracle_cache_after_step(w)
    qc = cs["qc"]
    cu = w.cu_seq_lens().numpy()
    ko, vo = oracle.gather_kv_cache_dequant(qc, np_i32(w.block_tables), np_i32(w.context_lens), cu,
                                            oracle.BF16 if out == "bf16" else oracle.F16)
    NB = qc.num_blocks
    ks = oracle.f16_bits_to_f64(qc.k_scale).transpose(0, 2, 1)            # [NB, 16, Hkv]
    k64 = (qc.k_q.astype(np.float64) * ks[..., None]).reshape(NB * 16, 2, 64)
    vs = np.repeat(oracle.f16_bits_to_f64(qc.v_scale).transpose(0, 2, 1, 3), 32, -1)
    vz = np.repeat(oracle.f16_bits_to_f64(qc.v_zero).transpose(0, 2, 1, 3), 32, -1)
    v64 = (_unpack_v(qc) * vs + vz).reshape(NB * 16, 2, 64)
    tdt = torch.bfloat16 if out == "bf16" else torch.float16
    table = np_i32(w.block_tables).astype(np.int64)
    for s in range(w.num_seqs):
        c = int(w.context_lens[s])
        t = np.arange(c)
        slots = table[s][t // 16] * 16 + t % 16
        for arr, got in ((k64, ko), (v64, vo)):
            ref = torch.from_numpy(arr[slots].astype(np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(got[cu[s]:cu[s] + c], ref)


def test_dequant_gather_of_fresh_quantisation_is_within_half_a_step():
    w = W.build(name="t", seed=10, context_lens=[33, 64], num_heads=4, num_kv_heads=2, head_dim=128,
                cache="k8v4", new_tokens="none")
    cs = oracle_cache_after_step(w)
    qc = cs["qc"]
    cu = w.cu_seq_lens().numpy()
    ko, vo = oracle.gather_kv_cache_dequant(qc, np_i32(w.block_tables), np_i32(w.context_lens), cu, oracle.F16)
    # history values in slot order -> logical order
    k_src = oracle.bf16_bits_to_f64(bits(w.k_hist))
    v_src = oracle.bf16_bits_to_f64(bits(w.v_hist))
    pos = {int(sl): i for i, sl in enumerate(np_i64(w.slot_hist))}
    table = np_i32(w.block_tables)
    for s in range(w.num_seqs):
        for t in range(int(w.context_lens[s])):
            i = pos[int(table[s, t // 16]) * 16 + t % 16]
            blk, off = int(table[s, t // 16]), t % 16
            kd = oracle.f16_bits_to_f64(ko[cu[s] + t])
            vd = oracle.f16_bits_to_f64(vo[cu[s] + t])
            sk = oracle.f16_bits_to_f64(qc.k_scale[blk, :, off])[:, None]
            sv = np.repeat(oracle.f16_bits_to_f64(qc.v_scale[blk, :, off]), 32, -1)
            ulp = np.abs(kd) * 2.0 ** -10 + 2.0 ** -24
            assert np.all(np.abs(kd - k_src[i]) <= 0.5 * sk * (1 + 2.0 ** -9) + ulp)
            lo = v_src[i].reshape(2, 4, 32).min(-1)
            vz = oracle.f16_bits_to_f64(qc.v_zero[blk, :, off])
            slack = np.repeat(np.abs(vz - lo) + 16 * np.abs(sv[:, ::32] - (v_src[i].reshape(2, 4, 32).max(-1) - lo) / 15), 32, -1)
            assert np.all(np.abs(vd - v_src[i]) <= 0.5 * sv + slack + np.abs(vd) * 2.0 ** -10 + 1e-7)


# ---------------------------------------------------------------- bytes model

def test_bytes_model_reproduces_the_pages_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_per_token.json")))
    per_tok = bytes_model.kv_bytes_per_token(g["n_layers"], g["kv_dim"], 1, g["bytes_per_elem"])
    assert per_tok == 131072                                  # 128 KiB
    tol = g["approx_rel_tolerance"]
    assert abs(per_tok - g["per_token_bytes_approx"]) <= tol * g["per_token_bytes_approx"]
    total = per_tok * g["context_tokens"]
    assert total == 4 * 2 ** 30                               # 4 GiB
    assert abs(total - g["context_bytes_approx"]) <= tol * g["context_bytes_approx"]


def test_k8v4_row_bytes():
    kb, vb = bytes_model.row_bytes("k8v4", 128)
    assert (kb, vb) == (130, 80)                # 128 codes + scale; 64 packed + 4 x (scale, zero)
    assert bytes_model.row_bytes("bf16", 128) == (256, 256)
