"""Compile libsgd (the CUDA sources under csrc/) for sm_103a, in tree.

The shared library lands next to this file as libsgd.so; object files go to
_build/.  Translation units compile in parallel; only what changed is rebuilt.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libsgd.so")
SOURCES = ["propose.cu", "backoff.cu", "corpus.cu", "sa_build.cu", "api.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsgd")


def _headers():
    hs = [os.path.join(INCLUDE, "sgd.h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _compile(src: str, flags) -> str:
    obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
    deps = [src] + _headers() + [os.path.abspath(__file__)]
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in deps):
        return obj
    tmp = obj + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-lineinfo", "-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
                             "-Xcompiler", "-fPIC", "-c", src, "-o", tmp] + list(flags)
    subprocess.check_call(cmd)
    os.replace(tmp, obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if force:
        for f in os.listdir(OUT_DIR):
            os.remove(os.path.join(OUT_DIR, f))
    flags = ["-Xptxas", "-v"] if verbose_ptxas else []
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with ThreadPoolExecutor(len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags), srcs))
    if (force or not os.path.exists(LIB_PATH)
            or os.path.getmtime(LIB_PATH) < max(os.path.getmtime(o) for o in objs)):
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build())
