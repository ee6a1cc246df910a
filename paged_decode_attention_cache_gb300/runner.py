"""One decode step of the paged attention path on the GPU, for a seeded workload.

A step is what one attention layer does per decode step: write the new
tokens' K/V into their cache slots (reshape_and_cache, or quantize_kv for the
K8/V4 cache), then attention over every sequence's visible tokens, either
single pass or split-KV followed by the log-sum-exp reduce.  All device
memory is allocated here by torch, once; the library itself allocates nothing.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import ops
from .workloads import Workload

_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}
F16_NAN = 0x7E00


def cascade_plan_for(w: Workload, min_members: int = 2, min_shared_blocks: int = 8):
    """The host grouping DecodeStep's cascade schedule uses: items of up to
    16 / g members (one tensor-core tile of query rows)."""
    width = max(1, 16 // (w.num_heads // w.num_kv_heads))
    return ops.pkv_cascade_plan(w.block_tables, w.context_lens, width, min_members=min_members,
                                min_shared_blocks=min_shared_blocks)


class DecodeStep:
    def __init__(self, w: Workload, device: str = "cuda", partition_size: Optional[int] = None,
                 out_dtype: Optional[torch.dtype] = None, schedule: Optional[str] = None,
                 cascade_min_members: int = 2, cascade_min_shared_blocks: int = 8):
        """schedule: "single" (one CTA per sequence and kv head), "split"
        (fixed partitions of partition_size tokens + LSE reduce) or "balanced"
        (equal block ranges per SM, combine fused) or "fused" (balanced, with the
        step's cache write in the same launch) or "cascade" (shared whole-page
        prefixes read once per group, balanced) or "sparse" (only the workload's
        listed pages, balanced); by default split when the workload names a
        partition size, else single."""
        self.w = w
        self.device = device
        dev = torch.device(device)
        self.partition_size = w.partition_size if partition_size is None else partition_size
        if schedule is None:
            schedule = "split" if self.partition_size > 0 else "single"
        if schedule not in ("single", "split", "balanced", "fused", "cascade", "sparse"):
            raise ValueError(schedule)
        if schedule != "split":
            self.partition_size = 0
        self.schedule = schedule
        self.seqs = ops.Seqs(w.block_tables.to(dev).contiguous(), w.context_lens.to(dev).contiguous(), w.q_len,
                             w.sliding_window)
        self.q = w.q.to(dev).contiguous()
        self.k_new = w.k_new.to(dev).contiguous()
        self.v_new = w.v_new.to(dev).contiguous()
        self.slot_new = w.slot_new.to(dev).contiguous()
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        if w.cache == "k8v4":
            self.cache = ops.Cache.empty("k8v4", w.num_blocks, w.num_kv_heads, w.head_dim, device=dev)
            nan = torch.tensor(F16_NAN, dtype=torch.int16).view(torch.float16).item()
            # slots never written keep NaN scales, so a stray read poisons the output
            self.cache.k_scale.fill_(nan)
            self.cache.v_scale.fill_(nan)
            self.cache.v_zero.fill_(nan)
            if w.k_hist is not None and w.k_hist.shape[0]:
                ops.pkv_quantize_kv(self.cache, w.k_hist.to(dev).contiguous(), w.v_hist.to(dev).contiguous(),
                                    w.slot_hist.to(dev).contiguous(), self.err)
        else:
            self.cache = ops.Cache(w.cache, w.k_cache.to(dev).contiguous().clone(),
                                   w.v_cache.to(dev).contiguous().clone())
        dt = out_dtype or _TORCH[w.src_dtype]
        self.out = torch.empty((w.num_rows, w.num_heads, w.head_dim), dtype=dt, device=dev)
        self.ws = None
        self.bal_ws = None
        if schedule == "split":
            nparts = -(-w.max_blocks * 16 // self.partition_size)
            self.ws = ops.split_workspace(w.num_rows, w.num_heads, w.head_dim, nparts, device=dev)
        elif schedule in ("balanced", "fused"):
            self.bal_ws = ops.balanced_workspace(w.num_seqs, w.num_kv_heads, w.head_dim, device=dev)
        elif schedule == "sparse":
            if w.page_lists is None:
                raise ValueError("the workload lists no pages")
            self.page_lists = w.page_lists.to(dev).contiguous()
            self.page_counts = w.page_counts.to(dev).contiguous()
            self.sparse_ws = ops.sparse_workspace(w.num_seqs, w.num_kv_heads, w.head_dim,
                                                  int(self.page_lists.shape[1]), device=dev)
        elif schedule == "cascade":
            if w.q_len != 1:
                raise ValueError("cascade attention is for q_len 1 decode")
            width = max(1, 16 // (w.num_heads // w.num_kv_heads))
            members, blocks = cascade_plan_for(w, cascade_min_members, cascade_min_shared_blocks)
            self.members = members.to(dev).contiguous()
            self.item_blocks = blocks.to(dev).contiguous()
            self.cascade_ws = ops.cascade_workspace(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                                    int(members.shape[0]), width, device=dev)

    @property
    def split(self) -> bool:
        return self.ws is not None

    def write(self, stream=None):
        if self.k_new.shape[0] == 0 or self.schedule == "fused":   # fused: written by the attention launch
            return
        if self.w.cache == "k8v4":
            ops.pkv_quantize_kv(self.cache, self.k_new, self.v_new, self.slot_new, self.err, stream)
        else:
            ops.pkv_reshape_and_cache(self.cache, self.k_new, self.v_new, self.slot_new, self.err, stream)

    def attend_phase1(self, stream=None):
        """The dominant kernel: single-pass / balanced attention, or split-KV phase 1."""
        if self.split:
            tmp, ml, es = self.ws
            ops.pkv_paged_attention_split(tmp, ml, es, self.partition_size, self.q, self.w.scale, self.cache,
                                          self.seqs, self.err, stream)
        elif self.schedule == "balanced":
            ops.pkv_paged_attention_balanced(self.out, self.q, self.w.scale, self.cache, self.seqs, self.bal_ws,
                                             self.err, stream)
        elif self.schedule == "sparse":
            ops.pkv_paged_attention_sparse(self.out, self.q, self.w.scale, self.cache, self.seqs, self.page_lists,
                                           self.page_counts, self.sparse_ws, self.err, stream)
        elif self.schedule == "cascade":
            ops.pkv_paged_attention_cascade(self.out, self.q, self.w.scale, self.cache, self.seqs, self.members,
                                            self.item_blocks, self.cascade_ws, self.err, stream)
        elif self.schedule == "fused":
            ops.pkv_decode_step_balanced(self.out, self.q, self.w.scale, self.cache, self.seqs, self.k_new,
                                         self.v_new, self.slot_new, self.bal_ws, self.err, stream)
        else:
            ops.pkv_paged_attention(self.out, self.q, self.w.scale, self.cache, self.seqs, self.err, stream)

    def attend_phase2(self, stream=None):
        if self.split:
            tmp, ml, es = self.ws
            ops.pkv_reduce(self.out, tmp, ml, es, self.seqs, self.partition_size, stream)

    def step(self, stream=None) -> torch.Tensor:
        self.write(stream)
        self.attend_phase1(stream)
        self.attend_phase2(stream)
        return self.out

    def launches_per_step(self) -> int:
        """Kernels of this library one step launches (clearing memsets not counted)."""
        wr = int(self.k_new.shape[0] > 0 and self.schedule != "fused")
        if self.schedule == "cascade":
            return wr + 3   # set-up, attention, reduce
        if self.schedule == "sparse":
            return wr + 2   # set-up, attention
        return wr + 1 + int(self.split)

    def gather(self, stream=None):
        """The visible tokens back as contiguous rows (K8/V4: dequantised to the source dtype)."""
        cu = self.w.cu_seq_lens().to(self.seqs.context_lens.device)
        total = int(cu[-1])
        k8v4 = self.w.cache == "k8v4"
        dt = _TORCH[self.w.src_dtype] if k8v4 else self.cache.k.dtype
        k_out = torch.empty((total, self.w.num_kv_heads, self.w.head_dim), dtype=dt, device=self.cache.k.device)
        v_out = torch.empty_like(k_out)
        if k8v4:
            ops.pkv_gather_kv_cache_dequant(k_out, v_out, cu, self.cache, self.seqs, self.err, stream)
        else:
            ops.pkv_gather_kv_cache(k_out, v_out, cu, self.cache, self.seqs, self.err, stream)
        return k_out, v_out

    def error_flags(self) -> int:
        return int(self.err.item())
