"""GPU parity of the dequantising gather (K8/V4 cache -> contiguous fp16/bf16):
bit-exact against the oracle, which forms each value in fp64, rounds it once to
fp32 and then to the output type.  Rows of tokens whose block id is bad are
left untouched and flagged."""
import numpy as np
import pytest
import torch

import oracle
from paged_decode_attention_cache_gb300 import ops, workloads as W
from paged_decode_attention_cache_gb300.runner import DecodeStep
from tests.helpers import bits, np_i32, oracle_cache_after_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_decode_attention_cache_gb300 import build
    build.build()
    ops.lib()
    torch.cuda.set_device(0)


def _check(w):
    st = DecodeStep(w, "cuda", partition_size=0)
    st.write()
    k_out, v_out = st.gather()
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    qc = oracle_cache_after_step(w)["qc"]
    ko, vo = oracle.gather_kv_cache_dequant(qc, np_i32(w.block_tables), np_i32(w.context_lens),
                                            w.cu_seq_lens().numpy(),
                                            oracle.BF16 if w.src_dtype == "bf16" else oracle.F16)
    assert np.array_equal(bits(k_out), ko)
    assert np.array_equal(bits(v_out), vo)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("Hkv", [1, 2, 8])
def test_dequant_gather_bit_exact(D, src, Hkv):
    w = W.build(name="t", seed=700 + D + Hkv, context_lens=[1, 15, 16, 17, 100, 0, 513], num_heads=2 * Hkv,
                num_kv_heads=Hkv, head_dim=D, cache="k8v4", src_dtype=src, value_scale=3.0)
    _check(w)


def test_dequant_gather_k8v4_batch32():
    _check(W.k8v4_batch32(device="cuda"))


def test_dequant_gather_rejects_fp16_caches_and_bad_dtype():
    w = W.build(name="t", seed=1, context_lens=[20], num_heads=4, num_kv_heads=2, head_dim=64, cache="f16",
                device="cuda")
    st = DecodeStep(w, "cuda", partition_size=0)
    k = torch.empty((20, 2, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(ops.PkvError):
        ops.pkv_gather_kv_cache_dequant(k, torch.empty_like(k), w.cu_seq_lens().cuda(), st.cache, st.seqs)
