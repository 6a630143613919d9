"""Builds libxs.so (the C-ABI library) in-tree with nvcc for sm_103a.

Translation units are compiled in parallel into ``_build/`` at the repository
root and linked into ``all_layout_gb300/libxs.so`` (CUDA runtime linked
statically; the driver's tensor-map encoder is fetched at run time).
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libxs.so")
SOURCES = ("attn.cu", "scatter.cu", "api.cu", "noalloc.cu", "probe.cu")
HEADERS = (os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "internal.h"),
           os.path.join(CSRC, "attn_wide.cuh"),
           os.path.join(ROOT, "include", "xs.h"))
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
NVCC_FLAGS = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden"]


# Sources of the attention kernel and its launch path: their hash names the kernel
# build that a measurement or an ncu summary was taken on.
KERNEL_SOURCES = ("attn.cu", "ptx.cuh", "internal.h", "api.cu", "attn_wide.cuh")


def kernel_sha() -> str:
    """First 16 hex digits of the SHA-256 over the kernel sources, in order."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(CSRC, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = [os.path.join(BUILD_DIR, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    todo = []
    for src, obj in zip(SOURCES, objs):
        path = os.path.join(CSRC, src)
        if force or _stale(obj, (path,) + HEADERS):
            todo.append([nvcc(), *NVCC_FLAGS, "-c", path, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, todo))
    if force or todo or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([nvcc(), ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
