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
