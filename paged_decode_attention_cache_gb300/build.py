"""Builds libpkv.so (the CUDA library behind include/pkv.h) in-tree with nvcc.

Each translation unit is compiled for sm_103a only, in parallel, then linked
into one shared library with the CUDA runtime linked statically.  A rebuild
happens only when a source or header is newer than the library.

``build(timeline=True)`` builds the same sources with -DPKV_TIMELINE into
libpkv_timeline.so: the attention kernels then stamp %globaltimer at fixed
points into a buffer that ``timeline.py`` reads.  Nothing else loads it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libpkv.so")
OBJDIR = os.path.join(PKG, "_build")
LIB_TIMELINE = os.path.join(PKG, "libpkv_timeline.so")
OBJDIR_TIMELINE = os.path.join(PKG, "_build_timeline")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, timeline: bool = False) -> str:
    lib, objdir = (LIB_TIMELINE, OBJDIR_TIMELINE) if timeline else (LIB, OBJDIR)
    if not force and not stale(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if timeline:
        extra += ["-DPKV_TIMELINE"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for (_, log), src in zip(results, srcs):
            if log.strip():
                print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    objs = [o for o, _ in results]
    tmp = lib + f".tmp.{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
