"""GPU parity of cascade attention [mlxcel manual "KV Cache", §"Paged Decode
Storage and Kernels": cascade attention for groups sharing a whole-page
prefix].  Cascade is a schedule, not a new operation: its output must equal
plain paged decode attention, so the oracle is the oracle's paged_attention on
the same cache, at the fp16/bf16 and K8/V4 tolerances of the other parity
tests.  Groups share physical blocks through their block tables; the pool's
unwritten slots are NaN, so a read past a prefix or a context shows."""
import numpy as np
import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import ALL_CORES, guard, oracle_attention
from tests.test_gpu_parity import check_attention

pytestmark = pytest.mark.gpu

K8V4_ABS = 2e-2
PKV_DEVERR_CASCADE = 0x10


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


def run_cascade(w, min_shared=1):
    st = DecodeStep(w, "cuda", out_dtype=torch.float32, schedule="cascade", cascade_min_shared_blocks=min_shared)
    g = guard(st)
    out = st.step()
    torch.cuda.synchronize()
    assert st.error_flags() == 0, f"device error flags {st.error_flags():#x}"
    g.check()
    return st, out.double().cpu().numpy()


GROUPS = [[0, 1, 2, 3, 4], [5, 6], [8, 9, 10]]
CTX = [81, 100, 300, 97, 81, 90, 200, 50, 81, 81, 700, 17]


@pytest.mark.parametrize("shared", [1, 5, 8])
@pytest.mark.parametrize("dt,H,Hkv,D", [("bf16", 32, 8, 128), ("f16", 4, 4, 64), ("bf16", 16, 2, 128),
                                        ("f16", 8, 1, 64)])
def test_cascade_decode(shared, dt, H, Hkv, D):
    ctx = [c + 16 * (shared - 5) if c > 80 else c for c in CTX]
    w = W.build(name="t", seed=700 + H + D + shared, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                cache=dt, prefix_groups=GROUPS, shared_blocks=shared)
    ref = oracle_attention(w, threads=8)
    st, got = run_cascade(w)
    assert st.members.shape[0] >= 3   # every group (or its cut) became an item
    check_attention(got, ref, False)


@pytest.mark.parametrize("H,Hkv", [(8, 2), (32, 8)])
def test_cascade_k8v4(H, Hkv):
    w = W.build(name="t", seed=710 + H, context_lens=CTX, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                cache="k8v4", prefix_groups=GROUPS, shared_blocks=5)
    ref = oracle_attention(w, threads=8)
    _, got = run_cascade(w)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= K8V4_ABS


def test_cascade_wide_group_and_empty_suffix():
    # group size 1: items of 16 members; members whose context ends on the
    # shared prefix have an empty suffix
    ctx = [64] * 5 + [65 + 7 * i for i in range(14)] + [30]
    w = W.build(name="t", seed=720, context_lens=ctx, num_heads=4, num_kv_heads=4, head_dim=64, cache="f16",
                prefix_groups=[list(range(19))], shared_blocks=4, new_tokens="none")
    ref = oracle_attention(w, threads=8)
    st, got = run_cascade(w)
    sizes = (st.members >= 0).sum(1).tolist()
    assert sorted(sizes) == [9, 10]
    check_attention(got, ref, False)


def test_cascade_no_items_is_plain_attention():
    w = W.build(name="t", seed=730, context_lens=[1, 16, 17, 300], num_heads=8, num_kv_heads=2, head_dim=128,
                cache="bf16")
    ref = oracle_attention(w, threads=8)
    st, got = run_cascade(w)
    assert st.members.shape[0] == 0
    check_attention(got, ref, False)


def test_cascade_bad_grouping_flags_and_stays_exact():
    """Members that cannot join (a different table, a context short of the
    prefix, a second item for the same sequence, an out-of-range index) are
    flagged and attended whole: the output still equals the oracle's."""
    ctx = [100, 120, 90, 40, 300, 81]
    w = W.build(name="t", seed=740, context_lens=ctx, num_heads=8, num_kv_heads=2, head_dim=128, cache="bf16",
                prefix_groups=[[0, 1, 2, 5]], shared_blocks=5)
    ref = oracle_attention(w, threads=8)
    st = DecodeStep(w, "cuda", out_dtype=torch.float32, schedule="split", partition_size=32)
    st.write()
    dev = st.q.device
    # item 0: 0, 1, 4 (table differs), 3 (context 40 < 80); item 1: 2, 0 (already
    # in item 0), 99 (out of range), -1 padding
    members = torch.tensor([[0, 1, 4, 3], [2, 0, 99, -1]], dtype=torch.int32, device=dev)
    blocks = torch.tensor([5, 5], dtype=torch.int32, device=dev)
    out = torch.empty_like(st.out)
    ws = ops.cascade_workspace(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, 2, 4, device=dev)
    ops.pkv_paged_attention_cascade(out, st.q, w.scale, st.cache, st.seqs, members, blocks, ws, st.err)
    torch.cuda.synchronize()
    assert st.error_flags() & PKV_DEVERR_CASCADE
    check_attention(out.double().cpu().numpy(), ref, False)


@pytest.mark.parametrize("out_dt", [torch.float16, torch.bfloat16])
def test_cascade_half_out(out_dt):
    w = W.build(name="t", seed=750, context_lens=CTX, num_heads=32, num_kv_heads=8, head_dim=128, cache="bf16",
                prefix_groups=GROUPS, shared_blocks=5)
    ref = oracle_attention(w, threads=8)
    st = DecodeStep(w, "cuda", out_dtype=out_dt, schedule="cascade", cascade_min_shared_blocks=1)
    got = st.step()
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    check_attention(got.double().cpu().numpy(), ref, True)


def test_cascade_serving_shape_full():
    """Batch 32 in 8 groups of 4 sharing a 2048-token prompt, own suffixes up to
    1024 tokens (the bench's cascade workload shape), every row."""
    w = W.cascade_b32_p2048(device="cpu")
    ref = oracle_attention(w, threads=ALL_CORES)
    st, got = run_cascade(w, min_shared=8)
    assert st.members.shape[0] == 8
    check_attention(got, ref, False)


def test_cascade_empty_and_one_token_sequences():
    # sequences with no token and with one token next to a shared group
    ctx = [0, 1, 81, 90, 100]
    w = W.build(name="t", seed=760, context_lens=ctx, num_heads=8, num_kv_heads=2, head_dim=64, cache="f16",
                prefix_groups=[[2, 3, 4]], shared_blocks=5, new_tokens="none")
    ref = oracle_attention(w, threads=8)
    st, got = run_cascade(w)
    assert st.members.shape[0] == 1
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    check_attention(got, ref, False)
