"""GPU parity of sliding-window decode: only the last W stored tokens of each
sequence are visible [MTPLX-2 §"Sliding-Window Memory Control"].  Every
schedule (single pass, fixed partitions + reduce, balanced) and every math
(CUDA-core decode, tensor-core verify, K8/V4) against the windowed oracle, with
the same tolerances as the unwindowed parity tests.  Pool slots outside the
stored context are NaN, so a read of anything the window or the context
excludes (beyond the masked tokens of a loaded block) shows in the output."""
import numpy as np
import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import ALL_CORES, oracle_attention, oracle_cache_after_step
from tests.test_gpu_parity import check_attention, run_step

pytestmark = pytest.mark.gpu

K8V4_ABS = 2e-2
CTX = [1, 15, 16, 17, 40, 100, 300]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("win", [1, 15, 16, 17, 37, 100, 4096])
@pytest.mark.parametrize("part", [0, 32, 64, "bal"])
@pytest.mark.parametrize("dt,H,Hkv,D", [("bf16", 8, 2, 128), ("f16", 4, 4, 64), ("bf16", 16, 2, 64)])
def test_window_decode(win, part, dt, H, Hkv, D):
    w = W.build(name="t", seed=400 + win + H, context_lens=CTX, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=dt, sliding_window=win)
    ref = oracle_attention(w, threads=8)
    _, got = run_step(w, part)
    check_attention(got, ref, False)


@pytest.mark.parametrize("win", [1, 17, 48, 4096])
@pytest.mark.parametrize("part", [0, 32, "bal"])
@pytest.mark.parametrize("dt,H,Hkv,ql", [("bf16", 8, 2, 4), ("f16", 16, 8, 2)])
def test_window_verify(win, part, dt, H, Hkv, ql):
    ctx = [4, 5, 16, 17, 100, 300]
    w = W.build(name="t", seed=500 + win + ql, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                cache=dt, q_len=ql, sliding_window=win)
    ref = oracle_attention(w, threads=8)
    _, got = run_step(w, part)
    check_attention(got, ref, False)


@pytest.mark.parametrize("win", [1, 17, 64, 4096])
@pytest.mark.parametrize("part", [0, 48, "bal"])
@pytest.mark.parametrize("H,Hkv,ql", [(8, 2, 1), (8, 2, 4)])
def test_window_k8v4(win, part, H, Hkv, ql):
    ctx = [4, 5, 17, 100, 300]
    w = W.build(name="t", seed=600 + win + ql, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                cache="k8v4", q_len=ql, sliding_window=win)
    cs = oracle_cache_after_step(w)
    ref = oracle_attention(w, cs, threads=8)
    _, got = run_step(w, part)
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= K8V4_ABS, f"max abs err {err:.3e}"


def test_window_split_partials_inside_the_window():
    """The fixed-partition partials the kernel writes are the oracle's partials
    for every partition the window reaches; the reduce combines only those."""
    P = 64
    w = W.build(name="t", seed=42, context_lens=[300, 70, 129], num_heads=8, num_kv_heads=2, head_dim=128,
                cache="bf16", sliding_window=100)
    cs = oracle_cache_after_step(w)
    NP = -(-w.max_blocks * 16 // P)
    ref, (po, pm, pl) = oracle_attention(w, cs, partition_size=P, max_partitions=NP, threads=8)
    st = DecodeStep(w, "cuda", partition_size=P)
    st.write()
    st.attend_phase1()
    torch.cuda.synchronize()
    tmp, ml, es = st.ws
    tmp = tmp.double().cpu().numpy(); ml = ml.double().cpu().numpy(); es = es.double().cpu().numpy()
    for s in range(w.num_seqs):
        ctx = int(w.context_lens[s])
        p0 = max(0, ctx - 100) // P
        for p in range(p0, -(-ctx // P)):
            np.testing.assert_allclose(tmp[s, :, p], po[s, :, p], atol=2e-3, rtol=1e-2)
            np.testing.assert_allclose(es[s, :, p], pl[s, :, p], rtol=1e-4)
            np.testing.assert_allclose(ml[s, :, p], pm[s, :, p], atol=1e-4)
    st.attend_phase2()
    torch.cuda.synchronize()
    check_attention(st.out.double().cpu().numpy(), ref, False)


def test_window_workload_full():
    """The sliding-window workload at full size, every row, balanced and split."""
    w = W.sliding_window_b8_w4096(device="cuda")
    st, got = run_step(w, "bal")
    ref = oracle_attention(w, threads=ALL_CORES)
    check_attention(got, ref, False)
    _, got_split = run_step(w, 512)
    check_attention(got_split, ref, False)


def test_negative_window_is_rejected():
    w = W.build(name="t", seed=1, context_lens=[20], num_heads=4, num_kv_heads=2, head_dim=64, cache="f16",
                device="cuda")
    st = DecodeStep(w, "cuda", partition_size=0)
    st.seqs.sliding_window = -1
    with pytest.raises(ops.PkvError):
        st.attend_phase1()
