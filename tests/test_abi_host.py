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
