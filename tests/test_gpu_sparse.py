"""GPU parity of sparse page-indirection decode [mlxcel manual "KV Cache",
§"Paged Decode Storage and Kernels": sparse page-indirection decode]: each
sequence attends only the stored tokens of the logical pages it lists, against
the oracle's sparse attention at the tolerances of the other parity tests.
Unlisted pages are never read: the pool's unwritten slots are NaN, and so are
the K/V of every unlisted page here, so a stray read shows."""
import numpy as np
import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import guard, oracle_attention, oracle_cache_after_step
from tests.test_gpu_parity import check_attention

pytestmark = pytest.mark.gpu

K8V4_ABS = 2e-2
PKV_DEVERR_PAGE_LIST = 0x20


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


def random_lists(seed, ctx, frac, max_pages=None, tail=None):
    rng = np.random.default_rng(seed)
    npg = [-(-c // 16) for c in ctx]
    mp = max_pages or max([1] + npg)
    pl = np.full((len(ctx), mp), -1, np.int32)
    pc = np.zeros(len(ctx), np.int32)
    for s, n in enumerate(npg):
        k = min(n, mp, int(round(frac * n)))
        sel = set(rng.choice(n, size=k, replace=False).tolist()) if n else set()
        if tail is not None and n:
            (sel.add if tail else sel.discard)(n - 1)
        sel = sorted(sel)[:mp]
        pl[s, :len(sel)] = sel
        pc[s] = len(sel)
    return torch.from_numpy(pl), torch.from_numpy(pc)


def poison_unlisted(w):
    """NaN into the K/V of every page a sequence does not list (fp16/bf16 pools)."""
    if w.cache == "k8v4":
        return
    for s in range(w.num_seqs):
        n = -(-int(w.context_lens[s]) // 16)
        keep = set(int(p) for p in w.page_lists[s, :int(w.page_counts[s])])
        for p in range(n):
            if p not in keep:
                pb = int(w.block_tables[s, p])
                w.k_cache[pb] = float("nan")
                w.v_cache[pb] = float("nan")


def run_sparse(w):
    st = DecodeStep(w, "cuda", out_dtype=torch.float32, schedule="sparse")
    g = guard(st)
    out = st.step()
    torch.cuda.synchronize()
    g.check()
    return st, out.double().cpu().numpy()


CTX = [1, 15, 16, 17, 40, 100, 300, 33]


@pytest.mark.parametrize("frac,tail", [(0.5, None), (0.3, True), (0.7, False), (1.0, None), (0.0, None)])
@pytest.mark.parametrize("dt,H,Hkv,D", [("bf16", 32, 8, 128), ("f16", 4, 4, 64), ("bf16", 16, 2, 128),
                                        ("f16", 8, 1, 64)])
def test_sparse_decode(frac, tail, dt, H, Hkv, D):
    w = W.build(name="t", seed=800 + H + D, context_lens=CTX, num_heads=H, num_kv_heads=Hkv, head_dim=D, cache=dt,
                new_tokens="none")
    w.page_lists, w.page_counts = random_lists(int(frac * 10) + H, CTX, frac, tail=tail)
    poison_unlisted(w)
    ref = oracle_attention(w, threads=8, sparse=True)
    st, got = run_sparse(w)
    assert st.error_flags() == 0, f"device error flags {st.error_flags():#x}"
    check_attention(got, ref, False)


def test_sparse_with_the_steps_write():
    # the new token's page (the tail) listed: the step's write reaches the attention
    w = W.build(name="t", seed=820, context_lens=CTX, num_heads=8, num_kv_heads=2, head_dim=128, cache="bf16")
    w.page_lists, w.page_counts = random_lists(3, CTX, 0.5, tail=True)
    ref = oracle_attention(w, threads=8, sparse=True)
    st, got = run_sparse(w)
    assert st.error_flags() == 0
    check_attention(got, ref, False)


@pytest.mark.parametrize("H,Hkv", [(8, 2), (32, 8)])
def test_sparse_k8v4(H, Hkv):
    w = W.build(name="t", seed=830 + H, context_lens=CTX, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                cache="k8v4")
    w.page_lists, w.page_counts = random_lists(7, CTX, 0.4, tail=True)
    ref = oracle_attention(w, threads=8, sparse=True)
    st, got = run_sparse(w)
    assert st.error_flags() == 0
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= K8V4_ABS


def test_sparse_bad_entries_flagged_and_skipped():
    ctx = [100, 64, 40]
    w = W.build(name="t", seed=840, context_lens=ctx, num_heads=8, num_kv_heads=2, head_dim=64, cache="f16",
                new_tokens="none")
    w.page_lists = torch.tensor([[0, 3, 3, 2, 6, 7, 99, -1], [5, 1, 2, 4, 0, 0, 0, 0], [-2, 0, 2, 1, 9, 0, 0, 0]],
                                dtype=torch.int32)
    w.page_counts = torch.tensor([8, 4, 5], dtype=torch.int32)
    ref = oracle_attention(w, threads=8, sparse=True)
    st, got = run_sparse(w)
    assert st.error_flags() & PKV_DEVERR_PAGE_LIST
    check_attention(got, ref, False)


def test_sparse_long_sequences_many_pages():
    # lists longer than a warp's 32 entries, several rounds of the compaction
    ctx = [4096, 2000, 700, 5000]
    w = W.build(name="t", seed=850, context_lens=ctx, num_heads=32, num_kv_heads=8, head_dim=128, cache="bf16",
                new_tokens="none")
    w.page_lists, w.page_counts = random_lists(9, ctx, 0.35)
    poison_unlisted(w)
    ref = oracle_attention(w, threads=16, sparse=True)
    st, got = run_sparse(w)
    assert st.error_flags() == 0
    check_attention(got, ref, False)


def test_sparse_32k_full():
    """The bench's sparse workload (batch 4 at 32K, a quarter of the pages)."""
    w = W.sparse_b4_32k(device="cpu")
    ref = oracle_attention(w, threads=16, sparse=True)
    st, got = run_sparse(w)
    assert st.error_flags() == 0
    check_attention(got, ref, False)


def test_sparse_empty_context_and_single_token():
    ctx = [0, 1, 33]
    w = W.build(name="t", seed=860, context_lens=ctx, num_heads=8, num_kv_heads=2, head_dim=64, cache="bf16",
                new_tokens="none")
    w.page_lists = torch.tensor([[0, 1, -1], [0, -1, -1], [0, 2, -1]], dtype=torch.int32)
    w.page_counts = torch.tensor([2, 1, 2], dtype=torch.int32)
    ref = oracle_attention(w, threads=8, sparse=True)
    st, got = run_sparse(w)
    # sequence 0 lists pages it does not have: skipped and flagged, zeros out
    assert st.error_flags() & PKV_DEVERR_PAGE_LIST
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    check_attention(got, ref, False)
