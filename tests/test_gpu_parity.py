"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bit-exact for cache writes, gathers and quantisation codes/scales; attention
within |gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise for fp16/bf16
outputs, and max-abs <= 2e-3 for fp32 outputs (fp32 accumulation against an
fp64 oracle over fp16/bf16 inputs).  Unused pool slots are NaN on both sides,
so any stray read fails the comparison.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import ALL_CORES, bits, guard, np_i32, np_i64, oracle_attention, oracle_cache_after_step

pytestmark = pytest.mark.gpu

ABS, REL = 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


def check_attention(got, ref, half_out):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), "non-finite GPU output"
    err = np.abs(got - ref)
    if half_out:
        bad = err > ABS + REL * np.abs(ref)
        assert not bad.any(), f"{bad.sum()} elements outside 2e-3 + 1e-2|ref| (max err {err.max():.3e})"
    else:
        assert err.max() <= ABS, f"max abs err {err.max():.3e}"
        big = np.abs(ref) >= 0.1
        if big.any():
            assert (err[big] / np.abs(ref[big])).max() <= REL
    return float(err.max())


def run_step(w, partition=None, out_dtype=torch.float32):
    """partition: None (workload default), 0 (single pass), P > 0 (split + reduce)
    or "bal" (balanced schedule with the fused combine)."""
    if partition == "bal":
        st = DecodeStep(w, "cuda", out_dtype=out_dtype, schedule="balanced")
    else:
        st = DecodeStep(w, "cuda", partition_size=partition, out_dtype=out_dtype)
    g = guard(st)
    out = st.step()
    torch.cuda.synchronize()
    assert st.error_flags() == 0, f"device error flags {st.error_flags():#x}"
    g.check()
    return st, out.double().cpu().numpy()


# ---------------------------------------------------------------- tiny fp16 step (64 tokens, 4 / 2 heads)

def test_tiny_f16_full_step():
    w = W.tiny_f16()
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs)
    for part in (0, 16, 32):
        st, got = run_step(w, part)
        check_attention(got, ref, False)
    assert np.array_equal(bits(st.cache.k), cs["k"]) and np.array_equal(bits(st.cache.v), cs["v"])
    k_out, v_out = st.gather()
    torch.cuda.synchronize()
    ko, vo = oracle.gather_kv_cache(cs["k"], cs["v"], np_i32(w.block_tables), np_i32(w.context_lens),
                                    w.cu_seq_lens().numpy())
    assert np.array_equal(bits(k_out), ko) and np.array_equal(bits(v_out), vo)
    st16, got16 = run_step(w, 0, torch.float16)
    check_attention(got16, ref, True)


# ---------------------------------------------------------------- small shapes, ragged edges

SMALL = []
for D in (64, 128):
    for H, Hkv in ((4, 4), (8, 4), (8, 2), (16, 2)):
        for dt in ("f16", "bf16"):
            SMALL.append((D, H, Hkv, dt))


@pytest.mark.parametrize("D,H,Hkv,dt", SMALL)
@pytest.mark.parametrize("part", [0, 16, 48, 512, "bal"])
def test_small_shapes(D, H, Hkv, dt, part):
    ctx = [0, 1, 15, 16, 17, 511, 512, 513]
    w = W.build(name="t", seed=100 + D + H, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=dt)
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=8)
    _, got = run_step(w, part)
    check_attention(got, ref, False)


def test_half_and_bf16_outputs():
    w = W.build(name="t", seed=5, context_lens=[33, 300], num_heads=8, num_kv_heads=2, head_dim=128,
                cache="bf16")
    ref = oracle_attention(w, threads=8)
    for dt in (torch.bfloat16, torch.float16):
        for part in (0, 64):
            _, got = run_step(w, part, dt)
            check_attention(got, ref, True)


# ---------------------------------------------------------------- full-size workloads

def test_llama3_8b_batch8_full():
    w = W.llama3_8b_batch8(device="cuda")
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=ALL_CORES)
    for part in (256, 0, "bal"):
        st, got = run_step(w, part)
        check_attention(got, ref, False)
    # the write touched exactly the new tokens' slots
    assert np.array_equal(bits(st.cache.k), cs["k"]) and np.array_equal(bits(st.cache.v), cs["v"])
    _, got_bf = run_step(w, 256, torch.bfloat16)
    check_attention(got_bf, ref, True)


def test_long_context_32k_split_and_partials():
    w = W.long_context_32k(device="cuda")
    cs = oracle_cache_after_step(w)
    NP = w.max_partitions
    ref, (po, pm, pl) = oracle_attention(w, cs, threads=ALL_CORES, partition_size=512, max_partitions=NP)
    st, got = run_step(w, 512)
    check_attention(got, ref, False)
    tmp, ml, es = (t.double().cpu().numpy() for t in st.ws)
    # partials: same partition outputs, and the same (m, l) up to where the max sits
    np.testing.assert_allclose(tmp, po, rtol=0, atol=ABS)
    lse_gpu = ml + np.log(es)
    lse_ref = pm + np.log(pl)
    np.testing.assert_allclose(lse_gpu, lse_ref, rtol=0, atol=1e-3)


def test_long_context_32k_balanced():
    w = W.long_context_32k(device="cuda")
    ref = oracle_attention(w, threads=ALL_CORES)
    _, got = run_step(w, "bal")
    check_attention(got, ref, False)


def test_balanced_many_ragged_sequences_and_workspace_reuse():
    """Hundreds of short and empty sequences: CTAs hold pieces of several
    sequences, pairs are cut across CTAs; the workspace counters return to zero
    and a second call on the same workspace gives the same bits."""
    rng = np.random.default_rng(3)
    ctx = [int(x) for x in rng.integers(0, 700, 300)]
    ctx[:5] = [0, 1, 16, 17, 0]
    w = W.build(name="t", seed=51, context_lens=ctx, num_heads=16, num_kv_heads=4, head_dim=128, cache="bf16")
    ref = oracle_attention(w, threads=16)
    st = DecodeStep(w, "cuda", out_dtype=torch.float32, schedule="balanced")
    out1 = st.step().clone()
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    check_attention(out1.double().cpu().numpy(), ref, False)
    n_pairs = w.num_seqs * w.num_kv_heads
    counters = st.bal_ws[-((n_pairs * 4 + 255) // 256 * 256):][: n_pairs * 4].view(torch.int32)
    assert int(counters.abs().sum()) == 0
    out2 = st.step()
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_reduce_kernel_on_oracle_partials():
    """The reduce alone, fed partials computed by the oracle."""
    w = W.build(name="t", seed=21, context_lens=[700, 1, 0, 1500], num_heads=8, num_kv_heads=2, head_dim=128,
                cache="bf16")
    cs = oracle_cache_after_step(w)
    P = 128
    NP = -(-w.max_blocks * 16 // P)
    _, (po, pm, pl) = oracle_attention(w, cs, partition_size=P, max_partitions=NP)
    ref = oracle.lse_reduce(po, pm, pl)
    seqs = ops.Seqs(w.block_tables.cuda(), w.context_lens.cuda(), 1)
    out = torch.empty((4, 8, 128), dtype=torch.float32, device="cuda")
    tmp = torch.from_numpy(po.astype(np.float32)).cuda()
    ml = torch.from_numpy(pm.astype(np.float32)).cuda()
    es = torch.from_numpy(pl.astype(np.float32)).cuda()
    ops.pkv_reduce(out, tmp, ml, es, seqs, P)
    torch.cuda.synchronize()
    check_attention(out.double().cpu().numpy(), ref, False)


# ---------------------------------------------------------------- quantiser

def test_quantize_kv_bit_exact_full_k8v4_workload():
    w = W.k8v4_batch32(device="cuda")
    st = DecodeStep(w, "cuda")
    st.write()
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    qc = oracle_cache_after_step(w)["qc"]
    c = st.cache
    assert np.array_equal(c.k.cpu().numpy(), qc.k_q)
    assert np.array_equal(c.v.cpu().numpy(), qc.v_q)
    assert np.array_equal(bits(c.k_scale), qc.k_scale)
    assert np.array_equal(bits(c.v_scale), qc.v_scale)
    assert np.array_equal(bits(c.v_zero), qc.v_zero)


@pytest.mark.parametrize("D,src", [(64, "f16"), (128, "f16"), (64, "bf16")])
def test_quantize_kv_bit_exact_small(D, src):
    w = W.build(name="t", seed=31, context_lens=[40, 17, 1], num_heads=4, num_kv_heads=4, head_dim=D,
                cache="k8v4", src_dtype=src, value_scale=3.0)
    st = DecodeStep(w, "cuda")
    st.write()
    torch.cuda.synchronize()
    qc = oracle_cache_after_step(w)["qc"]
    assert np.array_equal(st.cache.k.cpu().numpy(), qc.k_q)
    assert np.array_equal(st.cache.v.cpu().numpy(), qc.v_q)
    assert np.array_equal(bits(st.cache.k_scale), qc.k_scale)
    assert np.array_equal(bits(st.cache.v_scale), qc.v_scale)
    assert np.array_equal(bits(st.cache.v_zero), qc.v_zero)


# ---------------------------------------------------------------- device-side error reporting

def test_out_of_range_ids_are_flagged_not_fatal():
    w = W.build(name="t", seed=41, context_lens=[40, 40], num_heads=8, num_kv_heads=2, head_dim=128,
                cache="bf16")
    st = DecodeStep(w, "cuda", partition_size=0)
    st.seqs.block_tables[1, 1] = w.num_blocks + 7          # outside the pool
    st.slot_new[0] = w.num_blocks * 16 + 3                 # outside the pool
    st.step()
    torch.cuda.synchronize()
    flags = st.error_flags()
    assert flags & ops.DEVERR_OOB_BLOCK and flags & ops.DEVERR_OOB_SLOT
    assert torch.isfinite(st.out[0]).all()                  # the clean sequence is unaffected
    st.err.zero_()
    st.seqs.context_lens[0] = w.max_blocks * 16 + 5         # longer than its table
    st.attend_phase1()
    torch.cuda.synchronize()
    assert st.error_flags() & ops.DEVERR_CAPACITY


def test_host_validation_rejects_bad_arguments():
    w = W.tiny_f16(device="cuda")
    st = DecodeStep(w, "cuda", partition_size=32)
    tmp, ml, es = st.ws
    with pytest.raises(ops.PkvError) as ei:
        ops.pkv_paged_attention_split(tmp, ml, es, 24, st.q, w.scale, st.cache, st.seqs)
    assert ei.value.status == ops.PKV_ERR_INVALID_ARG
    with pytest.raises(ops.PkvError):
        ops.pkv_paged_attention(st.out, st.q.to(torch.bfloat16), w.scale, st.cache, st.seqs)
    bad = ops.Cache("f16", st.cache.k[:, :, :, :48].contiguous(), st.cache.v[:, :, :, :48].contiguous())
    with pytest.raises(ops.PkvError) as ei:
        ops.pkv_paged_attention(st.out, st.q, w.scale, bad, st.seqs)
    assert ei.value.status == ops.PKV_ERR_UNSUPPORTED
