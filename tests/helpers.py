"""Shared test plumbing: moving seeded workloads into the oracle's numpy form.

Nothing here computes attention or quantises: it converts tensors to raw bits
and calls the oracle."""
import numpy as np
import torch

import oracle

ODT = {"f16": oracle.F16, "bf16": oracle.BF16}
OCACHE = {"f16": oracle.CACHE_F16, "bf16": oracle.CACHE_BF16, "k8v4": oracle.CACHE_K8V4}


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 tensor as numpy uint16 (host copy)."""
    t = t.detach().cpu().contiguous()
    assert t.element_size() == 2
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def np_i32(t):
    return t.detach().cpu().contiguous().to(torch.int32).numpy().copy()


def np_i64(t):
    return t.detach().cpu().contiguous().to(torch.int64).numpy().copy()


def oracle_cache_after_step(w):
    """The oracle's own cache state after the step's write, built from the
    workload's inputs by the oracle's write routines."""
    if w.cache in ("f16", "bf16"):
        kc, vc = bits(w.k_cache), bits(w.v_cache)
        if w.k_new is not None and w.k_new.shape[0]:
            oracle.reshape_and_cache(kc, vc, bits(w.k_new), bits(w.v_new), np_i64(w.slot_new))
        return {"k": kc, "v": vc}
    qc = oracle.QuantCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.v_group)
    nan16 = np.uint16(0x7e00)
    qc.k_scale[:] = nan16       # unused slots poison any stray read
    qc.v_scale[:] = nan16
    qc.v_zero[:] = nan16
    odt = ODT[w.src_dtype]
    if w.k_hist is not None and w.k_hist.shape[0]:
        oracle.quantize_kv(qc, bits(w.k_hist), bits(w.v_hist), odt, np_i64(w.slot_hist))
    if w.k_new is not None and w.k_new.shape[0]:
        oracle.quantize_kv(qc, bits(w.k_new), bits(w.v_new), odt, np_i64(w.slot_new))
    return {"qc": qc}


def oracle_attention(w, cache_state=None, rows=None, threads=4, partition_size=0,
                     max_partitions=0, want_out=True, sparse=False):
    """sparse: attend only the workload's listed pages (page_lists / page_counts)."""
    cs = cache_state or oracle_cache_after_step(w)
    kw = dict(q_len=w.q_len, rows=rows, threads=threads, partition_size=partition_size,
              max_partitions=max_partitions, want_out=want_out, window=w.sliding_window)
    if sparse:
        kw.update(page_lists=np_i32(w.page_lists), page_counts=np_i32(w.page_counts))
    if w.cache == "k8v4":
        qc = cs["qc"]
        return oracle.paged_attention(bits(w.q), ODT[w.src_dtype], w.scale, oracle.CACHE_K8V4,
                                      qc.k_q, qc.v_q, np_i32(w.block_tables),
                                      np_i32(w.context_lens), k_scale=qc.k_scale,
                                      v_scale=qc.v_scale, v_zero=qc.v_zero, v_group=qc.v_group, **kw)
    return oracle.paged_attention(bits(w.q), ODT[w.src_dtype], w.scale, OCACHE[w.cache], cs["k"],
                                  cs["v"], np_i32(w.block_tables), np_i32(w.context_lens), **kw)
