"""Feeding a seeded workload to the oracle -- TEST INFRASTRUCTURE ONLY.

A workload (``paged_decode_attention_cache_gb300.workloads.Workload``, whose
module only draws inputs) is turned into the oracle's numpy form: raw 16-bit
patterns of q, K, V and the new tokens, int32 tables and lengths.  Then the
oracle's own routines build the cache state after the step's write
(reshape_and_cache, or quantize_kv over the history and the new tokens) and run
attention over it.  Nothing here computes attention, quantises or rounds: every
step of the method is a call into ``pkv_oracle.c``.  Like the rest of this
package it may be used only by the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg; this module never imports the CUDA library (it
reads the workload's tensors through their torch attributes only).
"""
from __future__ import annotations

import numpy as np

from . import (BF16, CACHE_BF16, CACHE_F16, CACHE_K8V4, F16, QuantCache, paged_attention,
               quantize_kv, reshape_and_cache)

ODT = {"f16": F16, "bf16": BF16}
OCACHE = {"f16": CACHE_F16, "bf16": CACHE_BF16, "k8v4": CACHE_K8V4}


def bits(t) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 torch tensor as numpy uint16 (host copy)."""
    import torch
    t = t.detach().cpu().contiguous()
    assert t.element_size() == 2
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def np_i32(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().to(torch.int32).numpy().copy()


def np_i64(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().to(torch.int64).numpy().copy()


def cache_after_step(w):
    """The oracle's own cache state after the step's write, built from the
    workload's inputs by the oracle's write routines."""
    if w.cache in ("f16", "bf16"):
        kc, vc = bits(w.k_cache), bits(w.v_cache)
        if w.k_new is not None and w.k_new.shape[0]:
            reshape_and_cache(kc, vc, bits(w.k_new), bits(w.v_new), np_i64(w.slot_new))
        return {"k": kc, "v": vc}
    qc = QuantCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.v_group)
    nan16 = np.uint16(0x7e00)
    qc.k_scale[:] = nan16       # unused slots poison any stray read
    qc.v_scale[:] = nan16
    qc.v_zero[:] = nan16
    odt = ODT[w.src_dtype]
    if w.k_hist is not None and w.k_hist.shape[0]:
        quantize_kv(qc, bits(w.k_hist), bits(w.v_hist), odt, np_i64(w.slot_hist))
    if w.k_new is not None and w.k_new.shape[0]:
        quantize_kv(qc, bits(w.k_new), bits(w.v_new), odt, np_i64(w.slot_new))
    return {"qc": qc}


def attention(w, cache_state=None, rows=None, threads=4, partition_size=0, max_partitions=0,
              want_out=True, sparse=False):
    """The oracle's attention over the workload (after its write).  rows: query
    rows to compute (others NaN); sparse: attend only the workload's listed
    pages (page_lists / page_counts)."""
    cs = cache_state or cache_after_step(w)
    kw = dict(q_len=w.q_len, rows=rows, threads=threads, partition_size=partition_size,
              max_partitions=max_partitions, want_out=want_out, window=w.sliding_window)
    if sparse:
        kw.update(page_lists=np_i32(w.page_lists), page_counts=np_i32(w.page_counts))
    if w.cache == "k8v4":
        qc = cs["qc"]
        return paged_attention(bits(w.q), ODT[w.src_dtype], w.scale, CACHE_K8V4, qc.k_q, qc.v_q,
                               np_i32(w.block_tables), np_i32(w.context_lens), k_scale=qc.k_scale,
                               v_scale=qc.v_scale, v_zero=qc.v_zero, v_group=qc.v_group, **kw)
    return paged_attention(bits(w.q), ODT[w.src_dtype], w.scale, OCACHE[w.cache], cs["k"], cs["v"],
                           np_i32(w.block_tables), np_i32(w.context_lens), **kw)
