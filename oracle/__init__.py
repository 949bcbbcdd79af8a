"""CPU fp64 attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``tiled_attention_forward_fwd_gb300``) never imports it and has no CPU
fallback.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows):
the materialised score row, batch softmax and weighted sum of V, exactly as the
lab 02 page's PyTorch reference ("Bloque C") and the standard-attention half of
the cruxr.ai worked example define attention.  This module only builds the
library with gcc and marshals arrays; it adds no arithmetic of its own beyond
the exact upcast of the stored fp16/bf16 inputs to float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` with gcc (-O2 -fopenmp, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci = ctypes.c_int
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ci, ci,
                                            ctypes.c_double, ci]
            lib.oracle_attn_fwd.restype = ci
            lib.oracle_attn_rows.argtypes = [dp, i64p, ctypes.c_long, dp, dp, dp, dp, ci, ci, ci,
                                             ci, ci, ci, ci, ci, ctypes.c_double, ci]
            lib.oracle_attn_rows.restype = ci
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().to(torch.float64).contiguous().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray, ct=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def attention(q, k, v, causal: bool = False, window: int = 0, sm_scale: float | None = None,
              nthreads: int = 0):
    """Full fp64 attention.  q: (B,Hq,Nq,d); k, v: (B,Hkv,Nk,d).

    Returns ``(O, LSE)`` as float64 numpy arrays of shapes (B,Hq,Nq,d) and
    (B,Hq,Nq)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    scale = float(sm_scale) if sm_scale is not None else 1.0 / float(np.sqrt(d))
    o = np.empty((B, Hq, Nq, d), dtype=np.float64)
    lse = np.empty((B, Hq, Nq), dtype=np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk,
                                 d, int(bool(causal)), int(window), scale, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd failed with code {rc}")
    return o, lse


def attention_rows(q_rows, row_ids, k, v, B: int, Hq: int, Nq: int, causal: bool = False,
                   window: int = 0, sm_scale: float | None = None, nthreads: int = 0):
    """fp64 attention for selected query rows only.

    ``row_ids`` are flat indices (b*Hq + h)*Nq + i; ``q_rows`` (n, d) are those
    rows of Q in the same order.  Returns ``(O_rows (n,d), LSE_rows (n,))``."""
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64))
    n, d = q_rows.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    scale = float(sm_scale) if sm_scale is not None else 1.0 / float(np.sqrt(d))
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_attn_rows(_ptr(q_rows), _ptr(ids, ctypes.c_int64), n, _ptr(k), _ptr(v),
                                  _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
                                  int(window), scale, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_rows failed with code {rc}")
    return o, lse
