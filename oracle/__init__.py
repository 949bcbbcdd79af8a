"""CPU fp64 attention oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``tiled_attention_forward_fwd_gb300``) never imports it and has no CPU
fallback.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows):
the materialised score row, batch softmax and weighted sum of V, exactly as the
lab 02 page's PyTorch reference ("Bloque C") and the standard-attention half of
the cruxr.ai worked example define attention; the gather through a page table;
and the gradients of that definition.  This module builds the library with gcc
and marshals arrays.  Its own arithmetic is limited to the exact upcast of the
stored fp16/bf16 inputs to float64, the latent cache's up-projections (one
numpy matrix product each, ``attention_mla``) and the INT8 cache's dequantising
multiply (``attention_kv_int8``), each followed by the C definition.
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
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_attn_paged.argtypes = [dp, dp, dp, i32p, i32p, dp, dp, ci, ci, ci, ci, ci, ci, ci,
                                              ci, ci, ci, ctypes.c_double, ci]
            lib.oracle_attn_paged.restype = ci
            lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ci, ci,
                                            ctypes.c_double]
            lib.oracle_attn_bwd.restype = ci
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


def attention_paged(q, k_pool, v_pool, block_table, seq_lens, causal: bool = False, window: int = 0,
                    sm_scale: float | None = None, nthreads: int = 0):
    """fp64 attention over a paged K/V cache.

    q: (B,Hq,Nq,d); k_pool, v_pool: (num_pages,Hkv,page_size,d); block_table:
    (B,max_pages) int; seq_lens: (B,) int.  Token t of request b is slot
    t % page_size of pool page block_table[b, t // page_size]; row i of
    request b sits at position seq_lens[b] - Nq + i.  Returns ``(O, LSE)``
    as float64 numpy arrays (B,Hq,Nq,d) and (B,Hq,Nq)."""
    q, kp, vp = _f64(q), _f64(k_pool), _f64(v_pool)
    if isinstance(block_table, torch.Tensor):
        block_table = block_table.cpu().numpy()
    if isinstance(seq_lens, torch.Tensor):
        seq_lens = seq_lens.cpu().numpy()
    table = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B, Hq, Nq, d = q.shape
    num_pages, Hkv, page_size = kp.shape[0], kp.shape[1], kp.shape[2]
    if vp.shape != kp.shape or kp.shape[3] != d or table.ndim != 2 or table.shape[0] != B or lens.shape != (B,):
        raise ValueError("paged oracle: inconsistent shapes")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / float(np.sqrt(d))
    o = np.empty((B, Hq, Nq, d), dtype=np.float64)
    lse = np.empty((B, Hq, Nq), dtype=np.float64)
    rc = _load().oracle_attn_paged(_ptr(q), _ptr(kp), _ptr(vp), _ptr(table, ctypes.c_int32),
                                   _ptr(lens, ctypes.c_int32), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, d,
                                   page_size, num_pages, table.shape[1], int(bool(causal)), int(window), scale,
                                   int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_paged failed with code {rc}")
    return o, lse


def attention_bwd(q, k, v, do, causal: bool = False, window: int = 0, sm_scale: float | None = None):
    """fp64 gradients of the forward definition for upstream gradient ``do``:
    returns ``(dQ, dK, dV)`` as float64 numpy arrays shaped like q, k, v (dK
    and dV summed over each kv head's query heads)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if do.shape != q.shape or v.shape != k.shape:
        raise ValueError("attention_bwd: inconsistent shapes")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / float(np.sqrt(d))
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv,
                                 Nq, Nk, d, int(bool(causal)), int(window), scale)
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd failed with code {rc}")
    return dq, dk, dv


def attention_mla(q, c, w_k_up, w_v_up, causal: bool = False, window: int = 0, sm_scale: float | None = None):
    """fp64 attention over a latent K/V cache (Multi-Head Latent Attention,
    cruxr.ai "Optimizaciones de Atencion", "Multi-Head Latent Attention
    (MLA)"): each token caches one vector c_t of d_c values, and keys and
    values are rebuilt per head by the up-projections
    K = c W_K^up, V = c W_V^up (W: d_c x (n_h * d_h)).

    q: (B, n_h, Nq, d_h); c: (B, Nk, d_c); w_k_up, w_v_up: (d_c, n_h * d_h).
    The keys and values of every head are decompressed explicitly (one matrix
    product each), then the plain definition runs as attention with n_h kv
    heads.  Returns ``(O, LSE)``, O (B, n_h, Nq, d_h)."""
    q, c, wk, wv = _f64(q), _f64(c), _f64(w_k_up), _f64(w_v_up)
    B, n_h, Nq, d_h = q.shape
    Nk, d_c = c.shape[1], c.shape[2]
    if c.shape[0] != B or wk.shape != (d_c, n_h * d_h) or wv.shape != wk.shape:
        raise ValueError("attention_mla: inconsistent shapes")
    k = (c @ wk).reshape(B, Nk, n_h, d_h).transpose(0, 2, 1, 3)
    v = (c @ wv).reshape(B, Nk, n_h, d_h).transpose(0, 2, 1, 3)
    return attention(q, k, v, causal=causal, window=window,
                     sm_scale=sm_scale if sm_scale is not None else 1.0 / float(np.sqrt(d_h)))


def attention_kv_int8(q, k_codes, v_codes, k_scale: float, v_scale: float, causal: bool = False, window: int = 0,
                      sm_scale: float | None = None):
    """fp64 attention over an INT8-quantised K/V cache (cruxr.ai
    "Optimizaciones de Atencion", "Elegir optimizaciones de atencion": INT8
    quantisation of the KV cache composes with the rest).  Symmetric codes
    with one fp32 scale per tensor: K = k_scale * k_codes, V = v_scale *
    v_codes (codes in [-127, 127]).  The cache is dequantised exactly in
    fp64, then the plain definition runs.  Returns ``(O, LSE)``."""
    kc, vc = _f64(k_codes), _f64(v_codes)
    if kc.shape != vc.shape or np.abs(kc).max(initial=0) > 127 or np.abs(vc).max(initial=0) > 127 or \
            not np.array_equal(kc, np.round(kc)) or not np.array_equal(vc, np.round(vc)):
        raise ValueError("attention_kv_int8: codes must be integers in [-127, 127] of equal shapes")
    if not (k_scale > 0 and v_scale > 0 and np.isfinite(k_scale) and np.isfinite(v_scale)):
        raise ValueError("attention_kv_int8: scales must be positive and finite")
    return attention(q, float(k_scale) * kc, float(v_scale) * vc, causal=causal, window=window, sm_scale=sm_scale)
