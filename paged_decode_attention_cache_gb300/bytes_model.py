"""Bytes a paged decode step must move: the algorithmic traffic the roofline is
measured against.

Decode attention reads every visible K and V row once per step, so its cost is
the size of the visible cache [metalworking, "The KV Cache": per token and
layer the cache holds one K and one V vector per kv head, and every decoded
token streams all of it].  The per-token growth is
``2 * n_layers * n_kv_heads * head_dim * bytes_per_elem`` [mlxcel manual, "KV
Cache", §"Memory Growth": the factor 2 counts K and V; the printed formula is
lost from the page, this is the reading the worked example fixes].
"""
from __future__ import annotations

BLOCK_SIZE = 16


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    """Cache bytes one token adds across all layers (K and V)."""
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def row_bytes(cache: str, head_dim: int, v_group: int = 32):
    """Bytes of one (token, kv head) K row and V row, metadata included."""
    if cache in ("f16", "bf16"):
        return 2 * head_dim, 2 * head_dim
    if cache == "k8v4":
        groups = head_dim // v_group
        return head_dim + 2, head_dim // 2 + 2 * 2 * groups
    raise ValueError(cache)


def attention_bytes(context_lens, q_len: int, num_heads: int, num_kv_heads: int, head_dim: int,
                    cache: str, q_bytes: int = 2, out_bytes: int = 2, v_group: int = 32,
                    sliding_window: int = 0) -> int:
    """K + V rows of every visible token, q in, out back, block table and lengths.

    K and V are counted once per (token, kv head): one CTA serves all query
    heads of a kv head, so a group's heads share the read.  With a sliding
    window only the last ``sliding_window`` stored tokens (and their blocks'
    table entries) count."""
    kb, vb = row_bytes(cache, head_dim, v_group)

    def span(c):
        c = int(c)
        lo = c - sliding_window if (sliding_window > 0 and c > sliding_window) else 0
        return lo, c

    kv = sum(c - lo for lo, c in map(span, context_lens)) * num_kv_heads * (kb + vb)
    rows = len(context_lens) * q_len
    qo = rows * num_heads * head_dim * (q_bytes + out_bytes)
    tables = 4 * sum(-(-c // BLOCK_SIZE) - lo // BLOCK_SIZE for lo, c in map(span, context_lens)) \
        + 4 * len(context_lens)
    return kv + qo + tables


def cascade_attention_bytes(context_lens, members, item_blocks, num_heads: int, num_kv_heads: int,
                            head_dim: int, cache: str, q_bytes: int = 2, out_bytes: int = 2,
                            v_group: int = 32) -> int:
    """Decode (q_len 1) with cascade items [mlxcel manual "KV Cache", §"Paged
    Decode Storage and Kernels"]: an item's shared blocks are read once for all
    its members, every sequence's own tokens after its item's prefix (all of
    them outside any item) once.  members: rows of sequence indices (< 0 pads),
    item_blocks: shared whole blocks per item, both as the planner returns them."""
    kb, vb = row_bytes(cache, head_dim, v_group)
    start = [0] * len(context_lens)
    prefix_tokens, prefix_blocks = 0, 0
    for row, nb in zip(members, item_blocks):
        nb = int(nb)
        prefix_tokens += nb * BLOCK_SIZE
        prefix_blocks += nb
        for m in row:
            if int(m) >= 0:
                start[int(m)] = nb * BLOCK_SIZE
    suffix_tokens = sum(int(c) - st for c, st in zip(context_lens, start))
    kv = (prefix_tokens + suffix_tokens) * num_kv_heads * (kb + vb)
    qo = len(context_lens) * num_heads * head_dim * (q_bytes + out_bytes)
    tables = 4 * (prefix_blocks + sum(-(-int(c) // BLOCK_SIZE) - st // BLOCK_SIZE
                                      for c, st in zip(context_lens, start))) + 4 * len(context_lens)
    return kv + qo + tables


def sparse_attention_bytes(context_lens, page_lists, page_counts, num_heads: int, num_kv_heads: int,
                           head_dim: int, cache: str, q_bytes: int = 2, out_bytes: int = 2,
                           v_group: int = 32) -> int:
    """Sparse page-indirection decode (q_len 1) [mlxcel manual "KV Cache",
    §"Paged Decode Storage and Kernels"]: K + V rows of the listed pages' stored
    tokens only, q in, out back, the list entries and the listed pages' block
    ids (read once, written compacted, read again), lengths.  Lists as the
    oracle reads them: in order, pages in range and above the last one taken."""
    kb, vb = row_bytes(cache, head_dim, v_group)
    tokens, pages, entries = 0, 0, 0
    for c, lst, n in zip(context_lens, page_lists, page_counts):
        c, n = int(c), int(n)
        npages, last = -(-c // BLOCK_SIZE), -1
        entries += n
        for p in list(lst)[:n]:
            p = int(p)
            if 0 <= p < npages and p > last:
                last = p
                pages += 1
                tokens += min(BLOCK_SIZE, c - p * BLOCK_SIZE)
    kv = tokens * num_kv_heads * (kb + vb)
    qo = len(context_lens) * num_heads * head_dim * (q_bytes + out_bytes)
    return kv + qo + 4 * entries + 3 * 4 * pages + 3 * 4 * len(context_lens)


def write_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, cache: str, src_bytes: int = 2,
                v_group: int = 32) -> int:
    """New K/V rows read from the source and written to their slots."""
    kb, vb = row_bytes(cache, head_dim, v_group)
    src = 2 * num_tokens * num_kv_heads * head_dim * src_bytes
    dst = num_tokens * num_kv_heads * (kb + vb)
    return src + dst + 8 * num_tokens


def split_overhead_bytes(num_rows: int, num_heads: int, head_dim: int, parts_written: int) -> int:
    """fp32 partials written by phase 1 and read back by the reduce (not counted
    as algorithmic bytes; reported separately)."""
    return 2 * parts_written * num_heads * (head_dim + 2) * 4
