"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every function include/pkv.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_decode_attention_cache_gb300 import build, ops
    build.build()
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(pkv_[a-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pkv_reshape_and_cache", "pkv_quantize_kv", "pkv_paged_attention", "pkv_paged_attention_split",
              "pkv_reduce", "pkv_gather_kv_cache", "pkv_split_workspace_bytes", "pkv_status_string",
              "pkv_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} missing from libpkv.so"


def test_product_library_has_no_timeline_stamps(lib):
    # the %globaltimer stamps (-DPKV_TIMELINE) live only in libpkv_timeline.so
    assert not hasattr(lib, "pkv_timeline_attach")


def test_status_strings(lib):
    for code, text in ((0, "ok"), (1, "invalid argument"), (2, "unsupported shape or type"), (3, "CUDA error")):
        assert lib.pkv_status_string(code).decode() == text


def test_workspace_size(lib):
    # tmp_out + max_logits + exp_sums, each padded to 256 bytes
    n = 8 * 32 * 16
    want = (n * 128 * 4 + 255) // 256 * 256 + 2 * ((n * 4 + 255) // 256 * 256)
    assert lib.pkv_split_workspace_bytes(8, 32, 128, 16) == want
    assert lib.pkv_split_workspace_bytes(0, 32, 128, 16) == 0


def test_null_arguments_rejected_without_a_gpu(lib):
    from paged_decode_attention_cache_gb300 import ops
    assert lib.pkv_paged_attention(None, 0, None, 0, 4, ctypes.c_float(0.1), None, None, None, None) == \
        ops.PKV_ERR_INVALID_ARG
    assert "cache is NULL" in lib.pkv_last_error().decode()
    c = ops._Cache(ops.PKV_CACHE_F16, 16, 16, 2, 64, 32, None, None, None, None, None)
    assert lib.pkv_reshape_and_cache(ctypes.byref(c), None, None, None, 1, None, None) == ops.PKV_ERR_INVALID_ARG
    c.block_size = 32
    assert lib.pkv_reshape_and_cache(ctypes.byref(c), None, None, None, 1, None, None) == ops.PKV_ERR_UNSUPPORTED
    assert "block_size" in lib.pkv_last_error().decode()
    # misaligned pointers are refused too
    c.block_size, c.k, c.v = 16, 0x1008, 0x2000
    assert lib.pkv_reshape_and_cache(ctypes.byref(c), None, None, None, 1, None, None) == ops.PKV_ERR_INVALID_ARG
    assert "aligned" in lib.pkv_last_error().decode()


def test_binding_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    from paged_decode_attention_cache_gb300 import build, ops
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        ops.lib()


def _valid_structs(ops, q_len=1, window=0, num_seqs=4, max_blocks=8):
    """A cache and a batch that pass the host checks; the device addresses are
    never dereferenced because every call below is refused first."""
    c = ops._Cache(ops.PKV_CACHE_BF16, 64, 16, 8, 128, 32, 0x10000, 0x20000, None, None, None)
    s = ops._Seqs(0x30000, 0x40000, num_seqs, max_blocks, q_len, window)
    return c, s


def _cascade(lib, c, s, members=0x50000, blocks=0x60000, items=2, width=4, ws=0x70000, ws_bytes=1 << 30,
             heads=32):
    return lib.pkv_paged_attention_cascade(0x80000, 1, 0x90000, 1, heads, ctypes.c_float(0.1), ctypes.byref(c),
                                           ctypes.byref(s), members, blocks, items, width, ws, ws_bytes, None,
                                           None)


def test_cascade_arguments_checked_on_the_host(lib):
    from paged_decode_attention_cache_gb300 import ops
    c, s = _valid_structs(ops, q_len=2)
    assert _cascade(lib, c, s) == ops.PKV_ERR_UNSUPPORTED and "q_len" in lib.pkv_last_error().decode()
    c, s = _valid_structs(ops, window=16)
    assert _cascade(lib, c, s) == ops.PKV_ERR_UNSUPPORTED and "window" in lib.pkv_last_error().decode()
    c, s = _valid_structs(ops)
    assert _cascade(lib, c, s, width=5) == ops.PKV_ERR_UNSUPPORTED          # 4 heads x 5 members > 16
    assert _cascade(lib, c, s, members=None) == ops.PKV_ERR_INVALID_ARG
    assert _cascade(lib, c, s, items=-1) == ops.PKV_ERR_INVALID_ARG
    need = lib.pkv_cascade_workspace_bytes(4, 32, 8, 128, 2, 4)
    assert need > 0
    assert _cascade(lib, c, s, ws_bytes=need - 1) == ops.PKV_ERR_INVALID_ARG
    assert "needs" in lib.pkv_last_error().decode()
    assert _cascade(lib, c, s, ws=0x70010) == ops.PKV_ERR_INVALID_ARG       # not 256-byte aligned
    assert _cascade(lib, c, s, ws=None) == ops.PKV_ERR_INVALID_ARG


def test_cascade_workspace_grows_with_items_and_rows(lib):
    base = lib.pkv_cascade_workspace_bytes(4, 32, 8, 128, 2, 4)
    assert lib.pkv_cascade_workspace_bytes(4, 32, 8, 128, 3, 4) >= base
    assert lib.pkv_cascade_workspace_bytes(8, 32, 8, 128, 2, 4) > base
    # two fp32 partials (o, max, sum) per row and head are part of it
    assert base >= 4 * 32 * 2 * (128 + 2) * 4
    assert lib.pkv_cascade_workspace_bytes(4, 32, 8, 128, 2, 17) == 0


def _sparse(lib, c, s, lists=0x50000, counts=0x60000, max_pages=8, ws=0x70000, ws_bytes=1 << 30):
    return lib.pkv_paged_attention_sparse(0x80000, 1, 0x90000, 1, 32, ctypes.c_float(0.1), ctypes.byref(c),
                                          ctypes.byref(s), lists, counts, max_pages, ws, ws_bytes, None, None)


def test_sparse_arguments_checked_on_the_host(lib):
    from paged_decode_attention_cache_gb300 import ops
    c, s = _valid_structs(ops, q_len=4)
    assert _sparse(lib, c, s) == ops.PKV_ERR_UNSUPPORTED and "q_len" in lib.pkv_last_error().decode()
    c, s = _valid_structs(ops, window=64)
    assert _sparse(lib, c, s) == ops.PKV_ERR_UNSUPPORTED
    c, s = _valid_structs(ops)
    assert _sparse(lib, c, s, max_pages=0) == ops.PKV_ERR_INVALID_ARG
    assert _sparse(lib, c, s, lists=None) == ops.PKV_ERR_INVALID_ARG
    assert _sparse(lib, c, s, counts=None) == ops.PKV_ERR_INVALID_ARG
    need = lib.pkv_sparse_workspace_bytes(4, 8, 128, 8)
    assert need == 256 + 256 + lib.pkv_balanced_workspace_bytes(4, 8, 128)   # compacted table + lengths + balanced
    assert _sparse(lib, c, s, ws_bytes=need - 1) == ops.PKV_ERR_INVALID_ARG
    assert _sparse(lib, c, s, ws=None) == ops.PKV_ERR_INVALID_ARG
