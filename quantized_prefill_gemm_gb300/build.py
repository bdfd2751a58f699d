"""Build the C-ABI shared library ``libq4k.so`` in-tree with nvcc (sm_103a).

Each translation unit compiles in parallel; the library is relinked only when
a source, header or flag changed (a content hash is kept beside the library),
so a stale binary is never picked up after a header edit.
"""
from __future__ import annotations

import hashlib
import re
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libq4k.so")
STAMP = LIB_PATH + ".stamp"

SOURCES = ["abi.cu", "act_quant.cu", "pack.cu", "gemm.cu", "gemv.cu", "gemv_stream.cu", "static_ws.cu", "peak.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put it on PATH)")


def _digest() -> str:
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/q4k.h"]
    for f in files:
        path = os.path.normpath(os.path.join(CSRC, f))
        if os.path.isfile(path):
            h.update(f.encode())
            with open(path, "rb") as fh:
                h.update(fh.read())
    # flags without the include paths, which are absolute and differ between checkouts
    h.update(" ".join(ARCH + [c for c in CFLAGS if not c.startswith("-I")] + SOURCES).encode())
    return h.hexdigest()


def _local_includes(src: str, csrc: str = CSRC) -> list:
    """src and every file of the directory csrc it includes, directly or not
    (#include "name" lines), in a fixed order."""
    seen, todo = [], [src]
    while todo:
        f = todo.pop(0)
        if f in seen or not os.path.exists(os.path.join(csrc, f)):
            continue
        seen.append(f)
        with open(os.path.join(csrc, f)) as fh:
            todo += re.findall(r'^\s*#include\s+"([^"/]+)"', fh.read(), flags=re.M)
    return seen


def _code_only(text: str) -> str:
    """C++ source without its comments and blank space (a comment edit does
    not change the kernel)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def gemm_digest(csrc: str = CSRC) -> str:
    """Hash of what the tensor-core GEMM kernel is built from: the code of
    gemm.cu and of the headers it includes (comments left out), and the
    flags.  Measurements of that kernel (the per-shape DRAM traffic table
    under profiles/) are keyed by it, so they stay valid while other kernels,
    or only comments, change."""
    h = hashlib.sha256()
    for f in _local_includes("gemm.cu", csrc):
        h.update(f.encode())
        with open(os.path.join(csrc, f)) as fh:
            h.update(_code_only(fh.read()).encode())
    h.update(" ".join(ARCH + [c for c in CFLAGS if not c.startswith("-I")]).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile and link; return the library path."""
    extra = list(extra_flags or [])
    digest = _digest() + ("|" + " ".join(extra) if extra else "")
    if not force and os.path.exists(LIB_PATH) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, res, cmd

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, _, res, cmd in results:
        if verbose or res.returncode:
            sys.stderr.write(res.stdout + res.stderr)
        if res.returncode:
            raise RuntimeError(f"nvcc failed on {src}: {' '.join(cmd)}")
    objs = [obj for _, obj, _, _ in results]
    tmp = LIB_PATH + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("link failed: " + " ".join(cmd))
    os.replace(tmp, LIB_PATH)
    with open(STAMP, "w") as f:
        f.write(digest)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
