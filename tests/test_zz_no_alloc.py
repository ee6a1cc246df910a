"""The allocation-free attention entry point (pkv_paged_attention_balanced_noalloc).

Some callers cannot allocate device memory: a plain C program that links only
this library has no device allocator of its own, and a serving loop with a fixed
memory budget must not allocate after start-up.  For them the library keeps its
balanced-schedule scratch in a static device array.  These tests call that entry
point through the C ABI, twice in a row on the same array, and check its output
against the entry point that takes a caller workspace: the two run the same
kernel with the same combine order, so their outputs must be identical bit for
bit.  One case is also checked against the oracle at the tolerances of the other
parity tests.  They run last (file name) so that a failure here never hides
another test, and they pass alone in a fresh process as well."""
import numpy as np
import pytest
import torch

from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import oracle_attention, oracle_cache_after_step

pytestmark = pytest.mark.gpu

ABS, REL = 2e-3, 1e-2
K8V4_ABS = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


def _reference(w):
    """Output of the workspace-taking entry point on the same inputs."""
    st = DecodeStep(w, "cuda", out_dtype=torch.float32, schedule="balanced")
    st.step()
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    return st, st.out.clone()


def _workload(name):
    if name == "llama3_8b_batch8":
        return W.llama3_8b_batch8(device="cuda")
    if name == "k8v4_small":
        return W.build(name="t", seed=61, context_lens=[40, 700, 3, 1500], num_heads=32, num_kv_heads=8,
                       head_dim=128, cache="k8v4")
    return W.build(name="t", seed=62, context_lens=[5, 900, 64, 2000], num_heads=16, num_kv_heads=4,
                   head_dim=128, cache="bf16", q_len=4)


def _noalloc_twice(w, st, ref):
    out = torch.empty_like(ref)
    for _ in range(2):   # the second call reuses the static array the first one left behind
        out.fill_(float("nan"))
        ops.pkv_paged_attention_balanced_noalloc(out, st.q, w.scale, st.cache, st.seqs, st.err)
        torch.cuda.synchronize()
        assert st.error_flags() == 0
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref), f"max diff {(out - ref).abs().max().item():.3e}"
    return out


@pytest.mark.parametrize("name", ["llama3_8b_batch8", "k8v4_small", "verify_small"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    w = _workload(name)
    st, ref = _reference(w)
    _noalloc_twice(w, st, ref)


def test_noalloc_against_the_oracle():
    """The verify-block case against the fp64 oracle, every row."""
    w = _workload("verify_small")
    st, ref = _reference(w)
    got = _noalloc_twice(w, st, ref).double().cpu().numpy()
    want = oracle_attention(w, oracle_cache_after_step(w), threads=8)
    err = np.abs(got - want)
    assert err.max() <= ABS and (err <= ABS + REL * np.abs(want)).all(), f"max err {err.max():.3e}"


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    B, H, Hkv, D = 4096, 32, 8, 128      # 32768 (sequence, kv head) pairs: far beyond 32 MiB of scratch
    need = ops.pkv_balanced_workspace_bytes(B, Hkv, D)
    assert need > 32 << 20
    cache = ops.Cache.empty("bf16", 4, Hkv, D)
    seqs = ops.Seqs(torch.zeros((B, 1), dtype=torch.int32, device="cuda"),
                    torch.zeros(B, dtype=torch.int32, device="cuda"), 1)
    q = torch.zeros((B, H, D), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, H, D), dtype=torch.float32, device="cuda")
    with pytest.raises(ops.PkvError) as ei:
        ops.pkv_paged_attention_balanced_noalloc(out, q, 0.1, cache, seqs)
    assert ei.value.status == ops.PKV_ERR_INVALID_ARG
    assert "static scratch" in str(ei.value)
