"""The C ABI from a plain C program (gcc, no CUDA headers): it compiles against
include/pkv.h, links libpkv.so and runs the host-only calls without a GPU."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_program_uses_the_abi(tmp_path):
    from paged_decode_attention_cache_gb300 import build
    lib = build.build()
    exe = tmp_path / "abi_host_example"
    src = os.path.join(ROOT, "tests", "c", "abi_host_example.c")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                        "-o", str(exe), lib, f"-Wl,-rpath,{os.path.dirname(lib)}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok ") >= 10
