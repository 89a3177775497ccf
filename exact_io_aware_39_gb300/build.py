"""Builds libflashattn.so in place from csrc/*.cu for sm_103a with nvcc.

The translation units are compiled in parallel and linked into one shared
library next to this file; objects go to _build/. Usage:
    python -m exact_io_aware_39_gb300.build [-v]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libflashattn.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_wide.cu", "fa_noalloc.cu", "std_attn.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-I", INCLUDE, "-I", CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            exe = cand
    if exe is None:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return exe


def link_flags():
    """cuBLAS (the plain GEMMs of the standard-attention baseline), found next
    to the nvcc in use and recorded as the library's run path."""
    cuda_home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    dirs = [d for d in (os.path.join(cuda_home, "lib64"), os.path.join(cuda_home, "lib")) if os.path.isdir(d)]
    flags = ["-lcublas"]
    for d in dirs:
        flags += ["-L", d, "-Xlinker", "-rpath=" + d]
    return flags


def _stale(obj, deps):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, extra_flags=()):
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    objs, procs = [], []
    for src in SOURCES:
        spath = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if _stale(obj, [spath, __file__] + headers):
            cmd = [nvcc(), *ARCH, *CFLAGS, *extra_flags, "-c", spath, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        text = out.decode(errors="replace")
        if pr.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            print(text)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if procs or not os.path.exists(LIB_PATH) or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, *link_flags()]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
