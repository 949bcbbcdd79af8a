"""Builds libattn.so (the C-ABI library of include/attn.h) in-tree with nvcc
for sm_103a.  Used by ``__graft_entry__.build()`` and on first import."""
from __future__ import annotations

import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libattn.so")
SOURCES = ["attn_api.cu"]
DEPS = ["attn_api.cu", "attn_fwd_sm103.cuh", "attn_bwd_sm103.cuh", "attn_decode.cuh", "attn_mla.cuh",
        "attn_short.cuh", "sm103_ptx.cuh", "fastdiv.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
_lock = threading.Lock()


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in DEPS] + [os.path.join(ROOT, "include", "attn.h")]
    return any(os.path.getmtime(f) > t for f in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    with _lock:
        if not force and not _stale():
            return LIB
        os.makedirs(LIBDIR, exist_ok=True)
        tmp = f"{LIB}.tmp{os.getpid()}"
        cmd = [_nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
               "-I", os.path.join(ROOT, "include"), "-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
        return LIB
