"""Python binding of libpkv.so (include/pkv.h) for torch tensors.

Argument marshalling only: every function checks dtypes, devices and
contiguity of the torch tensors it is given, passes their device pointers and
the current CUDA stream to the C entry point of the same name, and raises
``PkvError`` with the library's message on a non-OK status.  There is no CPU
path: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA = 0, 1, 2, 3
PKV_F16, PKV_BF16, PKV_F32 = 0, 1, 2
PKV_CACHE_F16, PKV_CACHE_BF16, PKV_CACHE_K8V4 = 0, 1, 2
DEVERR_OOB_BLOCK, DEVERR_OOB_SLOT, DEVERR_CAPACITY, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8

_DT = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.float32: PKV_F32}
_CACHE_KIND = {"f16": PKV_CACHE_F16, "bf16": PKV_CACHE_BF16, "k8v4": PKV_CACHE_K8V4}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status}: {message}")
        self.status = status


class _Cache(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("v_group", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p)]


class _Seqs(ctypes.Structure):
    _fields_ = [("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("sliding_window", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32


_lib_path: Optional[str] = None   # None: libpkv.so (build.LIB)


def library_path() -> str:
    return _lib_path or _build.LIB


def select_library(path: str) -> None:
    """Load another build of the same library (the timeline build) instead of
    libpkv.so; only before the first call."""
    global _lib_path
    if _lib is not None and path != library_path():
        raise RuntimeError("the library is already loaded")
    _lib_path = path


def lib():
    """Load libpkv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: call __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(path)
        st = ctypes.c_int
        L.pkv_reshape_and_cache.restype = st
        L.pkv_reshape_and_cache.argtypes = [_P, _P, _P, _P, _I32, _P, _P]
        L.pkv_quantize_kv.restype = st
        L.pkv_quantize_kv.argtypes = [_P, _P, _P, ctypes.c_int, _P, _I32, _P, _P]
        L.pkv_paged_attention.restype = st
        L.pkv_paged_attention.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, _I32, ctypes.c_float, _P, _P, _P, _P]
        L.pkv_split_workspace_bytes.restype = ctypes.c_size_t
        L.pkv_split_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
        L.pkv_paged_attention_split.restype = st
        L.pkv_paged_attention_split.argtypes = [_P, _P, _P, _I32, _I32, _P, ctypes.c_int, _I32, ctypes.c_float,
                                                _P, _P, _P, _P]
        L.pkv_reduce.restype = st
        L.pkv_reduce.argtypes = [_P, ctypes.c_int, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P]
        L.pkv_balanced_workspace_bytes.restype = ctypes.c_size_t
        L.pkv_balanced_workspace_bytes.argtypes = [_I32, _I32, _I32]
        L.pkv_paged_attention_balanced.restype = st
        L.pkv_paged_attention_balanced.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, _I32, ctypes.c_float, _P, _P,
                                                   _P, ctypes.c_size_t, _P, _P]
        L.pkv_decode_step_balanced.restype = st
        L.pkv_decode_step_balanced.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, _I32, ctypes.c_float, _P, _P,
                                               _P, _P, ctypes.c_int, _P, _I32, _P, ctypes.c_size_t, _P, _P]
        L.pkv_paged_attention_balanced_noalloc.restype = st
        L.pkv_paged_attention_balanced_noalloc.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, _I32, ctypes.c_float,
                                                           _P, _P, _P, _P]
        L.pkv_cascade_workspace_bytes.restype = ctypes.c_size_t
        L.pkv_cascade_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32]
        L.pkv_paged_attention_cascade.restype = st
        L.pkv_paged_attention_cascade.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, _I32, ctypes.c_float, _P, _P,
                                                  _P, _P, _I32, _I32, _P, ctypes.c_size_t, _P, _P]
        L.pkv_sparse_workspace_bytes.restype = ctypes.c_size_t
        L.pkv_sparse_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
        L.pkv_paged_attention_sparse.restype = st
        L.pkv_paged_attention_sparse.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, _I32, ctypes.c_float, _P, _P,
                                                 _P, _P, _I32, _P, ctypes.c_size_t, _P, _P]
        L.pkv_sparse_worthwhile.restype = _I32
        L.pkv_sparse_worthwhile.argtypes = [_P, _P, _I32, ctypes.c_float]
        L.pkv_cascade_plan.restype = st
        L.pkv_cascade_plan.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P]
        L.pkv_gather_kv_cache.restype = st
        L.pkv_gather_kv_cache.argtypes = [_P, _P, _P, _P, _P, _P, _P]
        L.pkv_gather_kv_cache_dequant.restype = st
        L.pkv_gather_kv_cache_dequant.argtypes = [_P, _P, ctypes.c_int, _P, _P, _P, _P, _P]
        L.pkv_status_string.restype = ctypes.c_char_p
        L.pkv_status_string.argtypes = [ctypes.c_int]
        L.pkv_last_error.restype = ctypes.c_char_p
        L.pkv_last_error.argtypes = []
        _lib = L
    return _lib


def _check(status: int):
    if status != PKV_OK:
        msg = lib().pkv_last_error().decode()
        raise PkvError(status, msg or lib().pkv_status_string(status).decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("pkv tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("pkv tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Cache:
    """One layer's paged cache (caller-owned device tensors)."""
    kind: str                 # "f16" | "bf16" | "k8v4"
    k: torch.Tensor           # [NB, 16, Hkv, D] (k8v4: int8)
    v: torch.Tensor           # [NB, 16, Hkv, D] (k8v4: uint8 [NB, 16, Hkv, D/2])
    k_scale: Optional[torch.Tensor] = None   # k8v4: fp16 [NB, Hkv, 16]
    v_scale: Optional[torch.Tensor] = None   # k8v4: fp16 [NB, Hkv, 16, D/32]
    v_zero: Optional[torch.Tensor] = None
    v_group: int = 32

    @property
    def num_blocks(self):
        return int(self.k.shape[0])

    @property
    def num_kv_heads(self):
        return int(self.k.shape[2])

    @property
    def head_dim(self):
        return int(self.k.shape[3])

    def c_struct(self) -> _Cache:
        return _Cache(_CACHE_KIND[self.kind], self.num_blocks, int(self.k.shape[1]), self.num_kv_heads,
                      self.head_dim, self.v_group, _ptr(self.k), _ptr(self.v), _ptr(self.k_scale),
                      _ptr(self.v_scale), _ptr(self.v_zero))

    @staticmethod
    def empty(kind: str, num_blocks: int, num_kv_heads: int, head_dim: int, device="cuda") -> "Cache":
        NB, H, D = num_blocks, num_kv_heads, head_dim
        if kind == "k8v4":
            return Cache(kind, torch.zeros((NB, 16, H, D), dtype=torch.int8, device=device),
                         torch.zeros((NB, 16, H, D // 2), dtype=torch.uint8, device=device),
                         torch.zeros((NB, H, 16), dtype=torch.float16, device=device),
                         torch.zeros((NB, H, 16, D // 32), dtype=torch.float16, device=device),
                         torch.zeros((NB, H, 16, D // 32), dtype=torch.float16, device=device))
        dt = torch.float16 if kind == "f16" else torch.bfloat16
        return Cache(kind, torch.zeros((NB, 16, H, D), dtype=dt, device=device),
                     torch.zeros((NB, 16, H, D), dtype=dt, device=device))


@dataclass
class Seqs:
    block_tables: torch.Tensor   # int32 [B, max_blocks]
    context_lens: torch.Tensor   # int32 [B]
    q_len: int = 1
    sliding_window: int = 0      # 0: none; W: only the last W stored tokens are visible

    def c_struct(self) -> _Seqs:
        if self.block_tables.dtype != torch.int32 or self.context_lens.dtype != torch.int32:
            raise ValueError("block_tables and context_lens must be int32")
        return _Seqs(_ptr(self.block_tables), _ptr(self.context_lens), int(self.block_tables.shape[0]),
                     int(self.block_tables.shape[1]), int(self.q_len), int(self.sliding_window))


def _err_ptr(err: Optional[torch.Tensor]):
    if err is None:
        return None
    if err.dtype not in (torch.int32, torch.uint32) or err.numel() < 1:
        raise ValueError("err_flags must be a device int32/uint32 tensor")
    return _ptr(err)


def pkv_reshape_and_cache(cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                          err_flags: Optional[torch.Tensor] = None, stream=None) -> None:
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    c = cache.c_struct()
    _check(lib().pkv_reshape_and_cache(ctypes.byref(c), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                       int(slot_mapping.numel()), _err_ptr(err_flags), _stream(stream)))


def pkv_quantize_kv(cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                    err_flags: Optional[torch.Tensor] = None, stream=None) -> None:
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    c = cache.c_struct()
    _check(lib().pkv_quantize_kv(ctypes.byref(c), _ptr(k_new), _ptr(v_new), _DT[k_new.dtype], _ptr(slot_mapping),
                                 int(slot_mapping.numel()), _err_ptr(err_flags), _stream(stream)))


def pkv_paged_attention(out: torch.Tensor, q: torch.Tensor, scale: float, cache: Cache, seqs: Seqs,
                        err_flags: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_paged_attention(_ptr(out), _DT[out.dtype], _ptr(q), _DT[q.dtype], int(q.shape[1]),
                                     float(scale), ctypes.byref(c), ctypes.byref(s), _err_ptr(err_flags),
                                     _stream(stream)))
    return out


def pkv_split_workspace_bytes(num_rows: int, num_heads: int, head_dim: int, max_partitions: int) -> int:
    return int(lib().pkv_split_workspace_bytes(num_rows, num_heads, head_dim, max_partitions))


def split_workspace(num_rows: int, num_heads: int, head_dim: int, max_partitions: int, device="cuda"):
    """Caller-side allocation of the split-KV scratch (torch owns it)."""
    tmp = torch.empty((num_rows, num_heads, max_partitions, head_dim), dtype=torch.float32, device=device)
    ml = torch.empty((num_rows, num_heads, max_partitions), dtype=torch.float32, device=device)
    es = torch.empty((num_rows, num_heads, max_partitions), dtype=torch.float32, device=device)
    return tmp, ml, es


def pkv_paged_attention_split(tmp_out, max_logits, exp_sums, partition_size: int, q: torch.Tensor, scale: float,
                              cache: Cache, seqs: Seqs, err_flags=None, stream=None) -> None:
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_paged_attention_split(_ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums), int(partition_size),
                                           int(tmp_out.shape[2]), _ptr(q), _DT[q.dtype], int(q.shape[1]),
                                           float(scale), ctypes.byref(c), ctypes.byref(s), _err_ptr(err_flags),
                                           _stream(stream)))


def pkv_reduce(out: torch.Tensor, tmp_out, max_logits, exp_sums, seqs: Seqs, partition_size: int,
               stream=None) -> torch.Tensor:
    s = seqs.c_struct()
    _check(lib().pkv_reduce(_ptr(out), _DT[out.dtype], _ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums),
                            ctypes.byref(s), int(tmp_out.shape[1]), int(tmp_out.shape[3]), int(partition_size),
                            int(tmp_out.shape[2]), _stream(stream)))
    return out


def pkv_balanced_workspace_bytes(num_seqs: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().pkv_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim))


def balanced_workspace(num_seqs: int, num_kv_heads: int, head_dim: int, device="cuda") -> torch.Tensor:
    """Caller-side, zero-filled scratch for pkv_paged_attention_balanced (torch owns it)."""
    n = pkv_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim)
    return torch.zeros(max(n, 1), dtype=torch.uint8, device=device)


def pkv_paged_attention_balanced(out: torch.Tensor, q: torch.Tensor, scale: float, cache: Cache, seqs: Seqs,
                                 workspace: torch.Tensor, err_flags: Optional[torch.Tensor] = None,
                                 stream=None) -> torch.Tensor:
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_paged_attention_balanced(_ptr(out), _DT[out.dtype], _ptr(q), _DT[q.dtype], int(q.shape[1]),
                                              float(scale), ctypes.byref(c), ctypes.byref(s), _ptr(workspace),
                                              int(workspace.numel() * workspace.element_size()),
                                              _err_ptr(err_flags), _stream(stream)))
    return out


def pkv_decode_step_balanced(out: torch.Tensor, q: torch.Tensor, scale: float, cache: Cache, seqs: Seqs,
                             k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                             workspace: torch.Tensor, err_flags: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """The step's cache write (reshape_and_cache / quantize_kv) and the balanced
    attention in one launch."""
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_decode_step_balanced(_ptr(out), _DT[out.dtype], _ptr(q), _DT[q.dtype], int(q.shape[1]),
                                          float(scale), ctypes.byref(c), ctypes.byref(s), _ptr(k_new), _ptr(v_new),
                                          _DT[k_new.dtype], _ptr(slot_mapping), int(slot_mapping.numel()),
                                          _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                          _err_ptr(err_flags), _stream(stream)))
    return out


def pkv_paged_attention_balanced_noalloc(out: torch.Tensor, q: torch.Tensor, scale: float, cache: Cache,
                                         seqs: Seqs, err_flags: Optional[torch.Tensor] = None,
                                         stream=None) -> torch.Tensor:
    """The balanced schedule with the library's own static scratch: for callers
    that cannot allocate device memory (see include/pkv.h for the size limit and
    the rule that calls sharing a device must not overlap)."""
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_paged_attention_balanced_noalloc(_ptr(out), _DT[out.dtype], _ptr(q), _DT[q.dtype],
                                                      int(q.shape[1]), float(scale), ctypes.byref(c),
                                                      ctypes.byref(s), _err_ptr(err_flags), _stream(stream)))
    return out


def pkv_cascade_plan(block_tables: torch.Tensor, context_lens: torch.Tensor, item_width: int,
                     min_members: int = 2, min_shared_blocks: int = 8):
    """Group sequences that share whole-page prefixes (host tensors in, host
    int32 tensors out): returns (members [num_items, item_width], item_blocks
    [num_items])."""
    bt = block_tables.detach().to("cpu", torch.int32).contiguous()
    cl = context_lens.detach().to("cpu", torch.int32).contiguous()
    n, mb = int(bt.shape[0]), int(bt.shape[1])
    if cl.numel() != n:
        raise ValueError("context_lens and block_tables disagree on num_seqs")
    cap = max(n // 2, 1)
    members = torch.full((cap, item_width), -1, dtype=torch.int32)
    blocks = torch.zeros(cap, dtype=torch.int32)
    count = ctypes.c_int32(0)
    _check(lib().pkv_cascade_plan(ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(cl.data_ptr()), n, mb,
                                  int(min_members), int(min_shared_blocks), int(item_width), cap,
                                  ctypes.c_void_p(members.data_ptr()), ctypes.c_void_p(blocks.data_ptr()),
                                  ctypes.byref(count)))
    k = int(count.value)
    return members[:k].clone(), blocks[:k].clone()


def pkv_cascade_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                num_items: int, item_width: int) -> int:
    return int(lib().pkv_cascade_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, num_items,
                                                 item_width))


def cascade_workspace(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, num_items: int,
                      item_width: int, device="cuda") -> torch.Tensor:
    """Caller-side scratch for pkv_paged_attention_cascade (needs no clearing)."""
    n = pkv_cascade_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, num_items, item_width)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


def pkv_paged_attention_cascade(out: torch.Tensor, q: torch.Tensor, scale: float, cache: Cache, seqs: Seqs,
                                members: torch.Tensor, item_blocks: torch.Tensor, workspace: torch.Tensor,
                                err_flags: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention with each item's shared prefix read once for all its
    members (device int32 members [num_items, width], item_blocks [num_items])."""
    if members.dtype != torch.int32 or item_blocks.dtype != torch.int32:
        raise ValueError("members / item_blocks must be int32")
    if members.dim() != 2 or item_blocks.numel() != members.shape[0]:
        raise ValueError("members must be [num_items, width] and item_blocks [num_items]")
    c, s = cache.c_struct(), seqs.c_struct()
    num_items, width = int(members.shape[0]), int(members.shape[1])
    _check(lib().pkv_paged_attention_cascade(_ptr(out), _DT[out.dtype], _ptr(q), _DT[q.dtype], int(q.shape[1]),
                                             float(scale), ctypes.byref(c), ctypes.byref(s),
                                             _ptr(members) if num_items else None,
                                             _ptr(item_blocks) if num_items else None, num_items,
                                             max(width, 1), _ptr(workspace),
                                             int(workspace.numel() * workspace.element_size()),
                                             _err_ptr(err_flags), _stream(stream)))
    return out


def pkv_sparse_workspace_bytes(num_seqs: int, num_kv_heads: int, head_dim: int, max_pages: int) -> int:
    return int(lib().pkv_sparse_workspace_bytes(num_seqs, num_kv_heads, head_dim, max_pages))


def sparse_workspace(num_seqs: int, num_kv_heads: int, head_dim: int, max_pages: int, device="cuda"):
    """Caller-side scratch for pkv_paged_attention_sparse (needs no clearing)."""
    n = pkv_sparse_workspace_bytes(num_seqs, num_kv_heads, head_dim, max_pages)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


def pkv_paged_attention_sparse(out: torch.Tensor, q: torch.Tensor, scale: float, cache: Cache, seqs: Seqs,
                               page_lists: torch.Tensor, page_counts: torch.Tensor, workspace: torch.Tensor,
                               err_flags: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention over the listed logical pages only (device int32
    page_lists [num_seqs, max_pages], page_counts [num_seqs])."""
    if page_lists.dtype != torch.int32 or page_counts.dtype != torch.int32:
        raise ValueError("page_lists / page_counts must be int32")
    if page_lists.dim() != 2 or page_counts.numel() != page_lists.shape[0]:
        raise ValueError("page_lists must be [num_seqs, max_pages] and page_counts [num_seqs]")
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_paged_attention_sparse(_ptr(out), _DT[out.dtype], _ptr(q), _DT[q.dtype], int(q.shape[1]),
                                            float(scale), ctypes.byref(c), ctypes.byref(s), _ptr(page_lists),
                                            _ptr(page_counts), int(page_lists.shape[1]), _ptr(workspace),
                                            int(workspace.numel() * workspace.element_size()),
                                            _err_ptr(err_flags), _stream(stream)))
    return out


def pkv_sparse_worthwhile(page_counts: torch.Tensor, context_lens: torch.Tensor, min_sparsity: float) -> bool:
    """Host policy: use sparse page-indirection when the lists leave out at least
    min_sparsity of all pages."""
    pc = page_counts.detach().to("cpu", torch.int32).contiguous()
    cl = context_lens.detach().to("cpu", torch.int32).contiguous()
    if pc.numel() != cl.numel():
        raise ValueError("page_counts and context_lens disagree on num_seqs")
    return bool(lib().pkv_sparse_worthwhile(ctypes.c_void_p(pc.data_ptr()), ctypes.c_void_p(cl.data_ptr()),
                                            int(pc.numel()), float(min_sparsity)))


def pkv_gather_kv_cache(k_out: torch.Tensor, v_out: torch.Tensor, cu_seq_lens: torch.Tensor, cache: Cache,
                        seqs: Seqs, err_flags=None, stream=None) -> None:
    if cu_seq_lens.dtype != torch.int32:
        raise ValueError("cu_seq_lens must be int32")
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_gather_kv_cache(_ptr(k_out), _ptr(v_out), _ptr(cu_seq_lens), ctypes.byref(c),
                                     ctypes.byref(s), _err_ptr(err_flags), _stream(stream)))


def pkv_gather_kv_cache_dequant(k_out: torch.Tensor, v_out: torch.Tensor, cu_seq_lens: torch.Tensor, cache: Cache,
                                seqs: Seqs, err_flags=None, stream=None) -> None:
    """K8/V4 cache -> contiguous fp16/bf16 (the dtype of k_out) K and V rows."""
    if cu_seq_lens.dtype != torch.int32:
        raise ValueError("cu_seq_lens must be int32")
    if k_out.dtype != v_out.dtype or k_out.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("k_out / v_out must both be float16 or both bfloat16")
    c, s = cache.c_struct(), seqs.c_struct()
    _check(lib().pkv_gather_kv_cache_dequant(_ptr(k_out), _ptr(v_out), _DT[k_out.dtype], _ptr(cu_seq_lens),
                                             ctypes.byref(c), ctypes.byref(s), _err_ptr(err_flags),
                                             _stream(stream)))
