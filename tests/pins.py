"""Independent CPU routines that pin the oracle (tests only).

None of these shares code with ``oracle/attn_oracle.c``; each reaches the
attention result by a different route, so a dropped term, a wrong sign, a
transposed operand or a wrong mask index in the oracle shows up as a mismatch.
"""
from __future__ import annotations

import math

import numpy as np


def live(p: int, j: int, causal: bool, window: int) -> bool:
    if causal and j > p:
        return False
    if window > 0 and p - j >= window:
        return False
    return True


def brute_attention(q, k, v, causal=False, window=0, sm_scale=None):
    """Pure-Python double loops with math.fsum (correctly rounded sums).

    q: nested lists / array (B,Hq,Nq,d); k, v: (B,Hkv,Nk,d).  Tiny sizes only."""
    q, k, v = np.asarray(q, float), np.asarray(k, float), np.asarray(v, float)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(d)
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            for i in range(Nq):
                p = Nk - Nq + i
                js = [j for j in range(Nk) if live(p, j, causal, window)]
                s = {j: scale * math.fsum(float(q[b, h, i, c]) * float(k[b, kh, j, c]) for c in range(d))
                     for j in js}
                M = max(s.values())
                w = {j: math.exp(s[j] - M) for j in js}
                l = math.fsum(w.values())
                for c in range(d):
                    O[b, h, i, c] = math.fsum(w[j] / l * float(v[b, kh, j, c]) for j in js)
                L[b, h, i] = M + math.log(l)
    return O, L


def tiled_online_attention(q, k, v, block_q=2, block_k=2, causal=False, window=0, sm_scale=None):
    """Tiled attention with the online-softmax recurrence, in fp64 numpy.

    Follows the steps of the cruxr.ai "FlashAttention" section: split Q into
    blocks of ``block_q`` rows and K/V into blocks of ``block_k`` rows; for each
    Q block keep a running maximum, a running sum of exponentials and an
    unnormalised output; for every K/V block rescale the running sum and output
    by exp(old_max - new_max), add the block's exponentials and weighted V rows;
    normalise once at the end.  The log-sum-exp is new_max + log(sum)."""
    q, k, v = np.asarray(q, float), np.asarray(k, float), np.asarray(v, float)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(d)
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    pos = np.arange(Nk)
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            for q0 in range(0, Nq, block_q):
                q1 = min(Nq, q0 + block_q)
                rows = np.arange(q0, q1)
                p = Nk - Nq + rows
                run_max = np.full(len(rows), -np.inf)
                run_sum = np.zeros(len(rows))
                acc = np.zeros((len(rows), d))
                for k0 in range(0, Nk, block_k):
                    k1 = min(Nk, k0 + block_k)
                    s = (q[b, h, q0:q1] @ k[b, kh, k0:k1].T) * scale
                    keep = np.ones_like(s, dtype=bool)
                    if causal:
                        keep &= pos[None, k0:k1] <= p[:, None]
                    if window > 0:
                        keep &= (p[:, None] - pos[None, k0:k1]) < window
                    s = np.where(keep, s, -np.inf)
                    new_max = np.maximum(run_max, s.max(axis=1))
                    safe = np.where(np.isfinite(new_max), new_max, 0.0)
                    corr = np.where(np.isfinite(run_max), np.exp(run_max - safe), 0.0)
                    w = np.where(keep, np.exp(s - safe[:, None]), 0.0)
                    run_sum = run_sum * corr + w.sum(axis=1)
                    acc = acc * corr[:, None] + w @ v[b, kh, k0:k1]
                    run_max = new_max
                O[b, h, q0:q1] = acc / run_sum[:, None]
                L[b, h, q0:q1] = run_max + np.log(run_sum)
    return O, L


def sin_matrix(rows: int, cols: int, seed: float):
    """Deterministic inputs of the cruxr.ai worked example: 0.5*sin(seed + i*cols + j)."""
    return [[math.sin(seed + i * cols + j) * 0.5 for j in range(cols)] for i in range(rows)]
