"""GPU parity of the tensor-core kernel: multi-token verify blocks on fp16/bf16
caches and the K8/V4 quantised cache, against the oracle (which dequantises
the same codes and scales exactly).

Tolerances: verify rows as for single-query decode (fp32 accumulation of
bf16/fp16 products); K8/V4 max-abs 2e-2 against the identically-dequantised
oracle (the kernel rounds q and p*scale_v to fp16 for the MMA)."""
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


def run(w, part, out_dtype=torch.float32):
    if part == "bal":
        st = DecodeStep(w, "cuda", out_dtype=out_dtype, schedule="balanced")
    else:
        st = DecodeStep(w, "cuda", partition_size=part, out_dtype=out_dtype)
    g = guard(st)
    out = st.step()
    torch.cuda.synchronize()
    assert st.error_flags() == 0, f"device error flags {st.error_flags():#x}"
    g.check()
    return st, out.double().cpu().numpy()


# ---------------------------------------------------------------- verify (q_len > 1)

# query rows per kv head (g * q_len): 16 (the 16-row tile), 8, 6 and 5 (the
# transposed tile, padding columns at 6 and 5), 3 (CUDA cores), and group size
# 8 decode (the transposed tile, 8 columns)
VERIFY = []
for D in (64, 128):
    for H, Hkv, ql in ((8, 2, 4), (32, 8, 4), (4, 4, 16), (16, 2, 2), (8, 2, 2), (8, 4, 3), (4, 4, 5), (8, 8, 3),
                       (16, 2, 1)):
        VERIFY.append((D, H, Hkv, ql))


@pytest.mark.parametrize("D,H,Hkv,ql", VERIFY)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("part", [0, 32, 512, "bal"])
def test_verify_small(D, H, Hkv, ql, dt, part):
    ctx = [2, 3, 4, 5, 16, 17, 100, 513]
    w = W.build(name="t", seed=200 + D + H + ql, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=dt, q_len=ql)
    ref = oracle_attention(w, threads=8)
    _, got = run(w, part)
    check_attention(got, ref, False)


def test_verify_batch256_full():
    """The serving-scale verify batch at full size: all 256 x 4 rows on the
    balanced, split and single-pass schedules (the oracle on every host core)."""
    w = W.verify_batch256(device="cuda")
    st, got = run(w, "bal")
    cs = oracle_cache_after_step(w)
    # the drafts' K/V were written by the step: whole pool bit-exact
    assert np.array_equal(bits(st.cache.k), cs["k"]) and np.array_equal(bits(st.cache.v), cs["v"])
    del st
    ref = oracle_attention(w, cs, threads=ALL_CORES)
    del cs
    check_attention(got, ref, False)
    _, got16 = run(w, 512, torch.bfloat16)
    check_attention(got16, ref, True)
    _, got_single = run(w, 0)
    check_attention(got_single, ref, False)


# ---------------------------------------------------------------- K8/V4

K8 = []
for D in (64, 128):
    for H, Hkv, ql in ((8, 2, 1), (32, 8, 1), (4, 4, 1), (16, 2, 1), (8, 2, 4)):
        K8.append((D, H, Hkv, ql))


@pytest.mark.parametrize("D,H,Hkv,ql", K8)
@pytest.mark.parametrize("part", [0, 48, 512, "bal"])
def test_k8v4_small(D, H, Hkv, ql, part):
    ctx = [1, 5, 16, 17, 100, 511, 513] if ql == 1 else [4, 5, 17, 100, 513]
    w = W.build(name="t", seed=300 + D + H + ql, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache="k8v4", q_len=ql)
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=8)
    st, got = run(w, part)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= K8V4_ABS, f"max abs err {err:.3e}"
    # the codes the kernel read are the oracle's codes
    qc = cs["qc"]
    assert np.array_equal(st.cache.k.cpu().numpy(), qc.k_q)
    assert np.array_equal(bits(st.cache.v_scale), qc.v_scale)


def test_k8v4_fp16_queries():
    w = W.build(name="t", seed=77, context_lens=[300, 40], num_heads=32, num_kv_heads=8, head_dim=128,
                cache="k8v4", src_dtype="f16")
    ref = oracle_attention(w, threads=8)
    _, got = run(w, 128)
    assert np.abs(got - ref).max() <= K8V4_ABS


def test_k8v4_batch32_full():
    """The K8/V4 batch at full size, all 32 rows, on the split, single-pass and
    balanced schedules."""
    w = W.k8v4_batch32(device="cuda")
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=ALL_CORES)
    for part in (512, 0, "bal"):
        _, got = run(w, part)
        assert np.isfinite(got).all()
        err = np.abs(got - ref).max()
        assert err <= K8V4_ABS, f"max abs err {err:.3e} (schedule {part})"
