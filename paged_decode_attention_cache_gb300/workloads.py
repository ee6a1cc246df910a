"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: block tables, context lengths, query/key/value
values and the slots new tokens are written to.  It holds none of the
attention, quantisation or reduction arithmetic, so both the CUDA library and
the CPU oracle can be fed from it without sharing any of the method's code.

Draw order (fixed, so a seed names one input set):
  context lengths of the named workloads: their own CPU generator, seeded ``seed + 7``
  structure generator (CPU, seeded with ``seed``):
    1. physical block permutation   2. spike-token mask
    3. free-slot choice (workloads whose new token goes outside the table)
  value generator (on ``device``, seeded with ``seed + 1000``):
    5. q   6. K pool   7. V pool   8. new-token K   9. new-token V
Values are drawn in fp32 and cast (round to nearest even) to the cache dtype.
Every pool slot that does not hold a visible history token is NaN (for fp16 /
bf16 caches), so a kernel that reads a slot it should not poisons its output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

BLOCK_SIZE = 16

_TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    cache: str                      # "f16" | "bf16" | "k8v4"
    src_dtype: str                  # dtype of q and of the K/V values ("f16" | "bf16")
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    q_len: int
    scale: float
    block_tables: torch.Tensor      # int32 [B, max_blocks], -1 past each sequence's blocks
    context_lens: torch.Tensor      # int32 [B], visible tokens including the new ones
    q: torch.Tensor                 # [B*q_len, H, D] src dtype
    # fp16/bf16 caches: the pool with history filled in, NaN elsewhere.
    k_cache: Optional[torch.Tensor] = None
    v_cache: Optional[torch.Tensor] = None
    # K8/V4 caches: history K/V as source values and their slots (quantised at set-up).
    k_hist: Optional[torch.Tensor] = None
    v_hist: Optional[torch.Tensor] = None
    slot_hist: Optional[torch.Tensor] = None
    # tokens written by every step (reshape_and_cache / quantize_kv)
    k_new: Optional[torch.Tensor] = None    # [T, Hkv, D]
    v_new: Optional[torch.Tensor] = None
    slot_new: Optional[torch.Tensor] = None  # int64 [T]
    partition_size: int = 0                  # 0: single pass
    sliding_window: int = 0                  # 0: every stored token is visible
    # sparse page-indirection decode: logical pages each sequence attends
    page_lists: Optional[torch.Tensor] = None   # int32 [B, max_pages]
    page_counts: Optional[torch.Tensor] = None  # int32 [B]
    block_size: int = BLOCK_SIZE
    v_group: int = 32
    notes: List[str] = field(default_factory=list)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_rows(self) -> int:
        return self.num_seqs * self.q_len

    @property
    def max_partitions(self) -> int:
        if self.partition_size <= 0:
            return 1
        return -(-self.max_blocks * self.block_size // self.partition_size)

    def cu_seq_lens(self) -> torch.Tensor:
        cu = torch.zeros(self.num_seqs + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(self.context_lens.cpu().to(torch.int64), 0).to(torch.int32)
        return cu


def _slots_of(table_row: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
    """Physical slot of each logical position: block_table[t // 16] * 16 + t % 16."""
    return table_row[positions // BLOCK_SIZE].to(torch.int64) * BLOCK_SIZE + positions % BLOCK_SIZE


def _randn(shape, gen, device, dtype, scale=1.0, chunk_rows=1 << 14):
    """fp32 N(0,1) draws cast to dtype, drawn in chunks along dim 0 to bound memory."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    for a in range(0, n0, chunk_rows):
        b = min(n0, a + chunk_rows)
        x = torch.randn((b - a,) + tuple(shape[1:]), generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        out[a:b] = x.to(dtype)
    return out


def build(*, name: str, seed: int, context_lens: List[int], num_heads: int, num_kv_heads: int,
          head_dim: int, cache: str = "bf16", src_dtype: Optional[str] = None, q_len: int = 1,
          num_blocks: Optional[int] = None, max_blocks: Optional[int] = None,
          new_tokens: str = "tail", value_scale: float = 1.0, spike_frac: float = 0.0,
          spike_scale: float = 8.0, partition_size: int = 0, identity_table: bool = False,
          device: str = "cpu", scale: Optional[float] = None, sliding_window: int = 0,
          prefix_groups: Optional[List[List[int]]] = None, shared_blocks: int = 0) -> Workload:
    """General seeded workload.

    new_tokens:
      "tail": the last ``q_len`` visible tokens of every sequence are new (written
              by the step); the rest is history.
      "free": one new token goes to a uniformly drawn slot of a block that no
              sequence owns; all visible tokens are history.
      "none": no new tokens.
    """
    src_dtype = src_dtype or ("bf16" if cache == "k8v4" else cache)
    tdt = _TORCH_DTYPES[src_dtype]
    B, H, Hkv, D, bs = len(context_lens), num_heads, num_kv_heads, head_dim, BLOCK_SIZE
    sgen = torch.Generator(device="cpu").manual_seed(seed)
    ctx = torch.tensor(context_lens, dtype=torch.int32)
    nblk = [(-(-c // bs)) for c in context_lens]
    # shared prefixes: the members of a group point their first shared_blocks
    # logical blocks at the same physical blocks (one copy of the prompt)
    group_of = {}
    for gi, members in enumerate(prefix_groups or []):
        for m in members:
            # the step's new token must land past the shared blocks
            assert context_lens[m] > shared_blocks * bs or (new_tokens != "tail" and
                                                            context_lens[m] == shared_blocks * bs), \
                "a member needs tokens past the shared prefix"
            group_of[m] = gi
    need = sum(nblk) - sum((len(mm) - 1) * shared_blocks for mm in (prefix_groups or []))
    if num_blocks is None:
        num_blocks = max(need + 1, int(math.ceil(1.1 * need)))
    if max_blocks is None:
        max_blocks = max(1, max(nblk) if nblk else 1)
    assert need <= num_blocks, "pool too small"
    # 1. physical block permutation: blocks handed out without replacement, sequence by sequence
    perm = torch.arange(num_blocks, dtype=torch.int32) if identity_table else \
        torch.randperm(num_blocks, generator=sgen).to(torch.int32)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    used = 0
    group_blocks = {}
    for s in range(B):
        first = 0
        if s in group_of:
            gi = group_of[s]
            if gi not in group_blocks:
                group_blocks[gi] = perm[used:used + shared_blocks]
                used += shared_blocks
            table[s, :shared_blocks] = group_blocks[gi]
            first = shared_blocks
        table[s, first:nblk[s]] = perm[used:used + nblk[s] - first]
        used += nblk[s] - first
    # 2. spike mask over every sequence's logical positions (peaked-softmax workloads)
    spikes = []
    if spike_frac > 0:
        for s in range(B):
            n = int(round(spike_frac * context_lens[s]))
            spikes.append(torch.randperm(context_lens[s], generator=sgen)[:n])
    # history / new split
    hist_pos, new_pos = [], []
    seen_group = set()
    for s in range(B):
        c = context_lens[s]
        # a shared prefix is history once (under its group's first member)
        h0 = 0
        if s in group_of:
            h0 = shared_blocks * bs if group_of[s] in seen_group else 0
            seen_group.add(group_of[s])
        if new_tokens == "tail":
            k = min(q_len, c)
            hist_pos.append(torch.arange(h0, c - k))
            new_pos.append(torch.arange(c - k, c))
        else:
            hist_pos.append(torch.arange(h0, c))
            new_pos.append(torch.arange(0, 0))
    slot_hist = torch.cat([_slots_of(table[s], hist_pos[s]) for s in range(B)]) if B else \
        torch.zeros(0, dtype=torch.int64)
    slot_new = torch.cat([_slots_of(table[s], new_pos[s]) for s in range(B)]) if B else \
        torch.zeros(0, dtype=torch.int64)
    if new_tokens == "free":
        free_blocks = perm[used:]
        assert free_blocks.numel() > 0, "no free block for the new token"
        # 3. free-slot choice
        b = int(torch.randint(free_blocks.numel(), (1,), generator=sgen))
        o = int(torch.randint(bs, (1,), generator=sgen))
        slot_new = torch.tensor([int(free_blocks[b]) * bs + o], dtype=torch.int64)

    vgen = torch.Generator(device=device).manual_seed(seed + 1000)
    R = B * q_len
    # 5. q
    q = _randn((R, H, D), vgen, device, tdt, value_scale)
    w = Workload(name=name, cache=cache, src_dtype=src_dtype, num_seqs=B, num_heads=H,
                 num_kv_heads=Hkv, head_dim=D, num_blocks=num_blocks, q_len=q_len,
                 scale=(1.0 / math.sqrt(D)) if scale is None else scale, block_tables=table,
                 context_lens=ctx, q=q, partition_size=partition_size, sliding_window=sliding_window)
    T = int(slot_new.numel())
    if cache in ("f16", "bf16"):
        # 6./7. K and V pools, then NaN everywhere but the history slots
        k_pool = _randn((num_blocks * bs, Hkv, D), vgen, device, tdt, value_scale)
        v_pool = _randn((num_blocks * bs, Hkv, D), vgen, device, tdt, value_scale)
        if spikes:
            for s in range(B):
                if spikes[s].numel():
                    sl = _slots_of(table[s], spikes[s]).to(device)
                    k_pool[sl] = (k_pool[sl].float() * spike_scale).to(tdt)
        keep = torch.zeros(num_blocks * bs, dtype=torch.bool, device=device)
        keep[slot_hist.to(device)] = True
        k_pool[~keep] = float("nan")
        v_pool[~keep] = float("nan")
        w.k_cache = k_pool.view(num_blocks, bs, Hkv, D)
        w.v_cache = v_pool.view(num_blocks, bs, Hkv, D)
    else:
        n_hist = int(slot_hist.numel())
        # 6./7. history K and V as source values for the quantiser
        w.k_hist = _randn((n_hist, Hkv, D), vgen, device, tdt, value_scale)
        w.v_hist = _randn((n_hist, Hkv, D), vgen, device, tdt, value_scale)
        w.slot_hist = slot_hist.to(device)
    # 8./9. new tokens
    w.k_new = _randn((T, Hkv, D), vgen, device, tdt, value_scale)
    w.v_new = _randn((T, Hkv, D), vgen, device, tdt, value_scale)
    w.slot_new = slot_new.to(device)
    w.block_tables = table.to(device)
    w.context_lens = ctx.to(device)
    return w


# --------------------------------------------------------------------------
# The five named workloads
# --------------------------------------------------------------------------

def _uniform_ints(gen, n, lo, hi):
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def tiny_f16(device="cpu", seed=0) -> Workload:
    """Batch 1, 4 query / 2 KV heads, head_dim 64, fp16, 64 tokens in 4 of 16 blocks;
    one new token written to a free slot, then gathered."""
    w = build(name="tiny_f16_b1_h4kv2_d64_ctx64", seed=seed, context_lens=[64], num_heads=4,
              num_kv_heads=2, head_dim=64, cache="f16", num_blocks=16, max_blocks=4,
              new_tokens="free", device=device)
    return w


def llama3_8b_batch8(device="cpu", seed=2, partition_size=256) -> Workload:
    """Llama-3-8B-like layer: batch 8, 32/8 heads, head_dim 128, bf16, pool 4096 blocks,
    context lengths uniform in [512, 4096], values N(0,1) * 0.5, one new token per sequence."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7)
    ctx = _uniform_ints(g, 8, 512, 4096)
    return build(name="llama3_8b_b8_h32kv8_d128_bf16", seed=seed, context_lens=ctx, num_heads=32,
                 num_kv_heads=8, head_dim=128, cache="bf16", num_blocks=4096, max_blocks=256,
                 value_scale=0.5, partition_size=partition_size, device=device)


def long_context_32k(device="cpu", seed=3) -> Workload:
    """Batch 1, context 32768 (2048 blocks of a 4096-block pool), 32/8 heads, head_dim 128,
    bf16, 1% of tokens with K scaled by 8, split into 512-token partitions."""
    return build(name="long32k_b1_h32kv8_d128_bf16_p512", seed=seed, context_lens=[32768],
                 num_heads=32, num_kv_heads=8, head_dim=128, cache="bf16", num_blocks=4096,
                 max_blocks=2048, new_tokens="none", spike_frac=0.01, spike_scale=8.0,
                 partition_size=512, device=device)


def k8v4_batch32(device="cpu", seed=4, partition_size=512) -> Workload:
    """Batch 32, 32/8 heads, head_dim 128, K int8 / V 4-bit cache, contexts uniform in
    [1024, 8192], N(0,1) bf16 sources; one new token per sequence quantised by the step."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7)
    ctx = _uniform_ints(g, 32, 1024, 8192)
    return build(name="k8v4_b32_h32kv8_d128", seed=seed, context_lens=ctx, num_heads=32,
                 num_kv_heads=8, head_dim=128, cache="k8v4", src_dtype="bf16", max_blocks=512,
                 partition_size=partition_size, device=device)


def verify_batch256(device="cpu", seed=5, partition_size=512) -> Workload:
    """Batch 256, 4 draft tokens per sequence (causal among themselves), 32/8 heads, head_dim
    128, bf16; context lengths lognormal (median 2048, sigma 1 on ln L) clipped to
    [128, 16384]; pool = blocks needed + 10%."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7)
    z = torch.randn(256, generator=g, dtype=torch.float64)
    ctx = [int(min(16384, max(128, round(2048.0 * math.exp(float(x)))))) for x in z]
    return build(name="verify_b256_q4_h32kv8_d128_bf16", seed=seed, context_lens=ctx,
                 num_heads=32, num_kv_heads=8, head_dim=128, cache="bf16", q_len=4,
                 max_blocks=1024, partition_size=partition_size, device=device)


def sliding_window_b8_w4096(device="cpu", seed=6, partition_size=512) -> Workload:
    """Sliding-window decode: batch 8, contexts uniform in [8192, 32768], only the last
    4096 stored tokens visible, 32/8 heads, head_dim 128, bf16, values N(0,1) * 0.5, one
    new token per sequence."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7)
    ctx = _uniform_ints(g, 8, 8192, 32768)
    return build(name="window4096_b8_h32kv8_d128_bf16", seed=seed, context_lens=ctx, num_heads=32,
                 num_kv_heads=8, head_dim=128, cache="bf16", max_blocks=2048, value_scale=0.5,
                 partition_size=partition_size, sliding_window=4096, device=device)


def cascade_b32_p2048(device="cpu", seed=7, partition_size=512) -> Workload:
    """Shared-prompt decode: batch 32 in 8 groups of 4 whose block tables point at the same
    128 physical blocks (a 2048-token prompt), each with its own suffix of uniform [16, 1024]
    tokens; 32/8 heads, head_dim 128, bf16, values N(0,1) * 0.5, one new token per sequence."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7)
    ctx = [2048 + x for x in _uniform_ints(g, 32, 16, 1024)]
    groups = [list(range(4 * i, 4 * i + 4)) for i in range(8)]
    return build(name="cascade_b32_g4_p2048_h32kv8_d128_bf16", seed=seed, context_lens=ctx, num_heads=32,
                 num_kv_heads=8, head_dim=128, cache="bf16", max_blocks=256, value_scale=0.5,
                 partition_size=partition_size, prefix_groups=groups, shared_blocks=128, device=device)


def sparse_pages(context_lens: List[int], seed: int, sink: int = 4, recent: int = 128,
                 middle_frac: float = 0.2, max_pages: Optional[int] = None):
    """Seeded page lists for sparse page-indirection decode: each sequence keeps
    its first `sink` pages, its last `recent` pages and a uniform random
    `middle_frac` of the pages between them (sorted, no repeats)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    npages = [-(-int(c) // BLOCK_SIZE) for c in context_lens]
    if max_pages is None:
        max_pages = max([1] + npages)
    lists = torch.full((len(context_lens), max_pages), -1, dtype=torch.int32)
    counts = torch.zeros(len(context_lens), dtype=torch.int32)
    for s, n in enumerate(npages):
        head = list(range(min(sink, n)))
        tail = list(range(max(len(head), n - recent), n))
        mid = list(range(len(head), tail[0] if tail else n))
        k = int(round(middle_frac * len(mid)))
        pick = sorted(mid[i] for i in torch.randperm(len(mid), generator=g)[:k].tolist()) if mid else []
        sel = head + pick + tail
        lists[s, :len(sel)] = torch.tensor(sel, dtype=torch.int32)
        counts[s] = len(sel)
    return lists, counts


def sparse_b4_32k(device="cpu", seed=8) -> Workload:
    """Sparse page-indirection decode at 32K: batch 4, context 32768 (2048 blocks each
    from an 8192+10% pool), 32/8 heads, head_dim 128, bf16, 1% of tokens with K x 8;
    each sequence attends its first 4 pages, its last 128 and 20% of the pages
    between (about 24% of the cache); one new token per sequence."""
    ctx = [32768] * 4
    w = build(name="sparse_b4_ctx32k_keep24_h32kv8_d128_bf16", seed=seed, context_lens=ctx, num_heads=32,
              num_kv_heads=8, head_dim=128, cache="bf16", max_blocks=2048, spike_frac=0.01,
              spike_scale=8.0, device=device)
    w.page_lists, w.page_counts = sparse_pages(ctx, seed + 11)
    return w


# every workload by name: the five decode / verify workloads of the scope, then
# those of the rows ranked next (windows, cascade prefixes, sparse page lists)
BY_NAME = {"tiny_f16": tiny_f16, "llama3_8b_batch8": llama3_8b_batch8, "long_context_32k": long_context_32k,
           "k8v4_batch32": k8v4_batch32, "verify_batch256": verify_batch256,
           "sliding_window_b8_w4096": sliding_window_b8_w4096, "cascade_b32_p2048": cascade_b32_p2048,
           "sparse_b4_32k": sparse_b4_32k}
