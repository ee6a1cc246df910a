"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper over ``pkv_oracle.c`` (plain scalar C, fp64).  Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the CUDA library never does, and this package never
imports the CUDA library.  All arrays are numpy; 16-bit floats travel as their
raw ``uint16`` bit patterns.

Pins (see ``tests/test_oracle_*.py``): number-format conversions against
numpy/torch conversions on sampled and edge-case bit patterns; attention against
closed forms (single token returns V, uniform keys return mean V), an
independent library attention (torch SDPA in fp64), paging invariants (identity
table equals a contiguous cache, permuting physical blocks changes nothing),
split-KV + LSE reduce equal to single pass, GQA equal to repeated kv heads,
verify-row causality equal to shorter single-query decodes; cache writes and
gathers against brute-force round trips; the quantiser against its error bounds
and hand-worked codes; the bytes model against the figures the pages print.
Unpinned: the pages' quoted K8/V4 cache size (6.21 GB -> 5.08 GB), which no
per-element format reproduces.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libpkv_oracle.so")

F16, BF16, F32, F64 = 0, 1, 2, 3
CACHE_F16, CACHE_BF16, CACHE_K8V4 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
             "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def use_library(path):
    """Point the wrapper at another build of the oracle (returns the previous
    handle); the mutation tests use it to run pins against planted mistakes."""
    global _lib
    prev = _lib
    if path is None:
        _lib = None
    else:
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return prev


def restore_library(handle):
    global _lib
    _lib = handle


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_D = ctypes.c_double


def _declare(L):
    L.pkvo_f16_to_f64.restype = _D
    L.pkvo_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.pkvo_bf16_to_f64.restype = _D
    L.pkvo_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.pkvo_f32_to_f16_rne.restype = ctypes.c_uint16
    L.pkvo_f32_to_f16_rne.argtypes = [ctypes.c_float]
    L.pkvo_f32_to_bf16_rne.restype = ctypes.c_uint16
    L.pkvo_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    for name in ("pkvo_f32_to_f16_array", "pkvo_f32_to_bf16_array",
                 "pkvo_f16_to_f64_array", "pkvo_bf16_to_f64_array"):
        fn = getattr(L, name)
        fn.restype = None
        fn.argtypes = [_P, _P, _I64]
    L.pkvo_reshape_and_cache.restype = _I
    L.pkvo_reshape_and_cache.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I]
    L.pkvo_gather_kv_cache.restype = _I
    L.pkvo_gather_kv_cache.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I]
    L.pkvo_quantize_kv.restype = _I
    L.pkvo_quantize_kv.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I]
    L.pkvo_paged_attention.restype = _I
    L.pkvo_paged_attention.argtypes = ([_P, _P, _P, _P, _I, _I, _P, _I, _I, _D, _I] + [_P] * 5 +
                                       [_I] * 5 + [_P, _P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _I])
    L.pkvo_gather_kv_cache_dequant.restype = _I
    L.pkvo_gather_kv_cache_dequant.argtypes = [_P, _P, _I, _P] + [_P] * 5 + [_P, _P] + [_I] * 7
    L.pkvo_lse_reduce.restype = None
    L.pkvo_lse_reduce.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().pkvo_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().pkvo_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().pkvo_f16_to_f64_array(_ptr(b), _ptr(out), b.size)
    return out


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().pkvo_bf16_to_f64_array(_ptr(b), _ptr(out), b.size)
    return out


def bits_to_f64(b: np.ndarray, dtype: int) -> np.ndarray:
    return f16_bits_to_f64(b) if dtype == F16 else bf16_bits_to_f64(b)


# --------------------------------------------------------------------------
# cache writes / reads
# --------------------------------------------------------------------------

def reshape_and_cache(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                      v_new: np.ndarray, slot_mapping: np.ndarray) -> int:
    """In place on k_cache / v_cache ([NB, bs, Hkv, D], any 2-byte dtype view).
    Returns the number of out-of-range slots skipped."""
    NB, bs, Hkv, D = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    slot = _c(slot_mapping, np.int64)
    return lib().pkvo_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                        _ptr(slot), slot.size, NB, bs, Hkv, D,
                                        k_cache.dtype.itemsize)


def gather_kv_cache(k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
                    context_lens: np.ndarray, cu_seq_lens: np.ndarray):
    NB, bs, Hkv, D = k_cache.shape
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    cu = _c(cu_seq_lens, np.int32)
    total = int(cu[-1])
    k_out = np.zeros((total, Hkv, D), k_cache.dtype)
    v_out = np.zeros((total, Hkv, D), v_cache.dtype)
    rc = lib().pkvo_gather_kv_cache(_ptr(k_out), _ptr(v_out), _ptr(cu), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(bt), _ptr(cl), bt.shape[0], bt.shape[1],
                                    NB, bs, Hkv, D, k_cache.dtype.itemsize)
    if rc:
        raise ValueError("oracle gather: out-of-range block id or context")
    return k_out, v_out


def gather_kv_cache_dequant(qc, block_tables: np.ndarray, context_lens: np.ndarray,
                            cu_seq_lens: np.ndarray, out_dtype: int = BF16):
    """K8/V4 codes -> contiguous [sum(ctx), Hkv, D] fp16/bf16 bits (uint16)."""
    NB, bs, Hkv, D = qc.k_q.shape
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    cu = _c(cu_seq_lens, np.int32)
    total = int(cu[-1])
    k_out = np.zeros((total, Hkv, D), np.uint16)
    v_out = np.zeros((total, Hkv, D), np.uint16)
    rc = lib().pkvo_gather_kv_cache_dequant(
        _ptr(k_out), _ptr(v_out), out_dtype, _ptr(cu), _ptr(qc.k_q), _ptr(qc.k_scale), _ptr(qc.v_q),
        _ptr(qc.v_scale), _ptr(qc.v_zero), _ptr(bt), _ptr(cl), bt.shape[0], bt.shape[1], NB, bs, Hkv, D,
        qc.v_group)
    if rc:
        raise ValueError("oracle dequantising gather: out-of-range block id or context")
    return k_out, v_out


class QuantCache:
    """K8/V4 cache arrays in the library's layout (numpy, host)."""

    def __init__(self, num_blocks, num_kv_heads, head_dim, block_size=16, v_group=32):
        NB, bs, H, D = num_blocks, block_size, num_kv_heads, head_dim
        self.k_q = np.zeros((NB, bs, H, D), np.int8)
        self.k_scale = np.zeros((NB, H, bs), np.uint16)
        self.v_q = np.zeros((NB, bs, H, D // 2), np.uint8)
        self.v_scale = np.zeros((NB, H, bs, D // v_group), np.uint16)
        self.v_zero = np.zeros((NB, H, bs, D // v_group), np.uint16)
        self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim = NB, bs, H, D
        self.v_group = v_group


def quantize_kv(qc: QuantCache, k_new: np.ndarray, v_new: np.ndarray, src_dtype: int,
                slot_mapping: np.ndarray) -> int:
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    slot = _c(slot_mapping, np.int64)
    return lib().pkvo_quantize_kv(_ptr(qc.k_q), _ptr(qc.k_scale), _ptr(qc.v_q), _ptr(qc.v_scale),
                                  _ptr(qc.v_zero), _ptr(k_new), _ptr(v_new), src_dtype, _ptr(slot),
                                  slot.size, qc.num_blocks, qc.block_size, qc.num_kv_heads,
                                  qc.head_dim, qc.v_group)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def paged_attention(q_bits: np.ndarray, q_dtype: int, scale: float, cache_kind: int,
                    k_cache, v_cache, block_tables, context_lens, q_len: int = 1,
                    k_scale=None, v_scale=None, v_zero=None, v_group: int = 32,
                    partition_size: int = 0, max_partitions: int = 0, rows=None,
                    threads: int = 1, want_out: bool = True, window: int = 0,
                    page_lists=None, page_counts=None):
    """fp64 paged attention.

    q_bits: [R, H, D] raw bits (uint16) for F16/BF16 (or float32/float64 with
    q_dtype F32/F64).  k_cache / v_cache: [NB, bs, Hkv, D] uint16 bits (f16/bf16
    caches) or the K8/V4 code arrays.  Returns ``out`` [R, H, D] (NaN in rows
    not computed when ``rows`` is given) and, if partition_size > 0,
    (part_o, part_m, part_l).  window > 0 keeps the last ``window`` stored
    tokens of each sequence visible (partitions wholly before them come back
    empty: o = 0, m = -inf, l = 0).  page_lists [B, max_pages] / page_counts [B]
    (int32): sparse page-indirection decode, each row attending only the tokens
    of its sequence's listed logical pages (no partitions).
    """
    q = np.ascontiguousarray(q_bits)
    R, H, D = q.shape
    if cache_kind == CACHE_K8V4:
        NB, bs, Hkv, _ = k_cache.shape
    else:
        NB, bs, Hkv, Dk = k_cache.shape
        assert Dk == D
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    assert R == bt.shape[0] * q_len
    out = np.full((R, H, D), np.nan) if want_out else None
    part = None
    if partition_size > 0:
        part = (np.zeros((R, H, max_partitions, D)), np.zeros((R, H, max_partitions)),
                np.zeros((R, H, max_partitions)))
    rl = None if rows is None else _c(np.asarray(rows, np.int32), np.int32)
    pl = pc = None
    if page_lists is not None:
        pl = _c(page_lists, np.int32)
        pc = _c(page_counts, np.int32)
        assert pl.ndim == 2 and pl.shape[0] == bt.shape[0] and pc.shape == (bt.shape[0],)
    rc = lib().pkvo_paged_attention(
        _ptr(out), _ptr(part[0]) if part else None, _ptr(part[1]) if part else None,
        _ptr(part[2]) if part else None, partition_size, max_partitions, _ptr(q), q_dtype, H,
        float(scale), cache_kind, _ptr(np.ascontiguousarray(k_cache)),
        _ptr(np.ascontiguousarray(v_cache)), _ptr(k_scale), _ptr(v_scale), _ptr(v_zero), NB, bs,
        Hkv, D, v_group, _ptr(bt), _ptr(cl), bt.shape[0], bt.shape[1], q_len, _ptr(rl),
        0 if rl is None else rl.size, threads, int(window), _ptr(pl), _ptr(pc),
        0 if pl is None else pl.shape[1])
    if rc:
        raise ValueError(f"oracle attention failed ({rc})")
    if part is not None:
        return out, part
    return out


def lse_reduce(part_o: np.ndarray, part_m: np.ndarray, part_l: np.ndarray) -> np.ndarray:
    part_o = _c(part_o, np.float64)
    part_m = _c(part_m, np.float64)
    part_l = _c(part_l, np.float64)
    R, H, P, D = part_o.shape
    out = np.zeros((R, H, D))
    lib().pkvo_lse_reduce(_ptr(out), _ptr(part_o), _ptr(part_m), _ptr(part_l), R, H, P, D)
    return out
