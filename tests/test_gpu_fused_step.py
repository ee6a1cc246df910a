"""GPU parity of the fused decode step (cache write + balanced attention in one
launch): the pool after the step is bit-exact against the oracle's write (or
quantisation), and the attention is within the tolerances of the unfused
calls, for fp16/bf16 decode, verify blocks, K8/V4 and sliding windows, with
new tokens written in place and elsewhere."""
import numpy as np
import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import ALL_CORES, bits, guard, oracle_attention, oracle_cache_after_step
from tests.test_gpu_parity import check_attention

pytestmark = pytest.mark.gpu

K8V4_ABS = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


def fused(w, out_dtype=torch.float32):
    st = DecodeStep(w, "cuda", schedule="fused", out_dtype=out_dtype)
    g = guard(st)
    out = st.step()
    torch.cuda.synchronize()
    assert st.error_flags() == 0, f"device error flags {st.error_flags():#x}"
    g.check()
    assert st.launches_per_step() == 1
    return st, out.double().cpu().numpy()


def check_pool(st, w, cs):
    if w.cache == "k8v4":
        qc = cs["qc"]
        assert np.array_equal(st.cache.k.cpu().numpy(), qc.k_q)
        assert np.array_equal(st.cache.v.cpu().numpy(), qc.v_q)
        assert np.array_equal(bits(st.cache.k_scale), qc.k_scale)
        assert np.array_equal(bits(st.cache.v_scale), qc.v_scale)
        assert np.array_equal(bits(st.cache.v_zero), qc.v_zero)
    else:
        assert np.array_equal(bits(st.cache.k), cs["k"]) and np.array_equal(bits(st.cache.v), cs["v"])


CASES = [
    # (cache, H, Hkv, D, q_len, new_tokens, window)
    ("bf16", 8, 2, 128, 1, "tail", 0),
    ("f16", 4, 4, 64, 1, "tail", 0),
    ("bf16", 32, 8, 128, 1, "tail", 0),
    ("bf16", 16, 2, 64, 1, "tail", 37),
    ("f16", 8, 1, 128, 1, "free", 0),
    ("bf16", 8, 2, 128, 4, "tail", 0),
    ("f16", 16, 8, 64, 2, "tail", 0),
    ("bf16", 8, 2, 128, 2, "tail", 0),
    ("bf16", 4, 2, 128, 3, "tail", 0),
    ("f16", 16, 2, 64, 1, "tail", 0),
    ("bf16", 8, 2, 128, 4, "tail", 48),
    ("k8v4", 8, 2, 128, 1, "tail", 0),
    ("k8v4", 32, 8, 128, 1, "tail", 0),
    ("k8v4", 8, 2, 64, 1, "tail", 17),
    ("k8v4", 8, 2, 128, 4, "tail", 0),
]


@pytest.mark.parametrize("cache,H,Hkv,D,ql,new,win", CASES)
def test_fused_step(cache, H, Hkv, D, ql, new, win):
    ctx = [4, 5, 16, 17, 33, 100, 300] if new == "tail" else [16, 17, 100]
    w = W.build(name="t", seed=900 + H + D + ql, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=cache, q_len=ql, new_tokens=new, sliding_window=win)
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=8)
    st, got = fused(w)
    check_pool(st, w, cs)
    if cache == "k8v4":
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= K8V4_ABS
    else:
        check_attention(got, ref, False)


def test_fused_step_tiny_free_slot():
    """The tiny workload's step (its default schedule): one new token written to a
    slot of a block the sequence does not own, then attention over the 64 tokens;
    the whole pool bit-exact, then the gather."""
    w = W.tiny_f16()
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs)
    st, got = fused(w)
    check_pool(st, w, cs)
    check_attention(got, ref, False)
    st16, got16 = fused(w, torch.float16)
    check_attention(got16, ref, True)


def test_fused_step_llama3_full():
    """The headline step at full size, every row, bf16 and fp32 outputs."""
    w = W.llama3_8b_batch8(device="cuda")
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=ALL_CORES)
    st, got = fused(w, torch.bfloat16)
    check_pool(st, w, cs)
    check_attention(got, ref, True)
    st, got32 = fused(w, torch.float32)
    check_pool(st, w, cs)
    check_attention(got32, ref, False)


def test_fused_step_k8v4_full():
    w = W.k8v4_batch32(device="cuda")
    cs = oracle_cache_after_step(w)
    st, got = fused(w)
    check_pool(st, w, cs)
    ref = oracle_attention(w, cs, threads=ALL_CORES)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= K8V4_ABS, f"max abs err {err:.3e}"


def test_fused_step_bad_slot_is_flagged_and_skipped():
    w = W.build(name="t", seed=5, context_lens=[40, 40], num_heads=8, num_kv_heads=2, head_dim=128, cache="bf16",
                new_tokens="free")
    st = DecodeStep(w, "cuda", schedule="fused")
    st.slot_new[0] = w.num_blocks * 16 + 3
    st.step()
    torch.cuda.synchronize()
    assert st.error_flags() & ops.DEVERR_OOB_SLOT
    assert torch.isfinite(st.out).all()


def test_fused_step_rejects_wrong_src_dtype():
    w = W.build(name="t", seed=6, context_lens=[20], num_heads=4, num_kv_heads=2, head_dim=64, cache="f16")
    st = DecodeStep(w, "cuda", schedule="fused")
    with pytest.raises(ops.PkvError):
        ops.pkv_decode_step_balanced(st.out, st.q, w.scale, st.cache, st.seqs, st.k_new.to(torch.bfloat16),
                                     st.v_new.to(torch.bfloat16), st.slot_new, st.bal_ws)
