"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI (via the thin binding), run the fp64 oracle on the same seeded inputs,
and compare element by element."""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import attn_inputs as ai

# Tolerances on O (max-abs vs the fp64 oracle) and LSE (abs), as stated for
# this path: fp16 I/O 1e-3, bf16 I/O 8e-3, LSE 1e-3.
TOL_O = {"fp16": 1e-3, "bf16": 8e-3}
TOL_LSE = 1e-3


def dtype_ulp(dtype: str, x: np.ndarray) -> np.ndarray:
    """Spacing of the 16-bit output grid at |x| (fp16: 11 significant bits,
    bf16: 8)."""
    bits = 11 if dtype == "fp16" else 8
    tiny = 2.0 ** -14 if dtype == "fp16" else 2.0 ** -126
    ax = np.maximum(np.abs(x), tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - (bits - 1))


# Unit roundoff of the 16-bit probability P fed to the P V contraction
# (round-to-nearest: half the spacing at 1, i.e. 2^-11 for fp16's 11
# significant bits and 2^-8 for bf16's 8).
U_P = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def o_tolerance(dtype: str, o_ref: np.ndarray, a_ref: np.ndarray | None = None) -> np.ndarray:
    """Elementwise bound on |O_gpu - O_oracle| (O_oracle unrounded fp64).

    The stated bound (1e-3 for fp16 I/O, 8e-3 for bf16 I/O) holds wherever the
    arithmetic the pages prescribe can meet it.  That arithmetic rounds each
    probability to the value dtype before P V (lab 02: ``p.to(v.dtype)``) and
    stores O in that dtype, so an exact kernel following it is off by up to
        u_P * sum_j w_j |V_jc|            (rounded probabilities)
      + half an ulp of the output         (rounded O)
      + a few fp32 roundings              (accumulation, exp2, 1/l)
    with w the exact softmax weights.  ``a_ref`` = sum_j w_j |V_jc| is the
    oracle run on |V|.  The bound applied is the larger of the stated one and
    this derived one."""
    stated = np.full_like(o_ref, TOL_O[dtype])
    if a_ref is None:
        return np.maximum(stated, dtype_ulp(dtype, o_ref))
    derived = U_P[dtype] * a_ref * (1.0 + 2.0 ** -10) + 0.5 * dtype_ulp(dtype, np.abs(o_ref) + U_P[dtype] * a_ref) \
        + 1e-5 * (np.abs(o_ref) + a_ref) + 1e-6
    return np.maximum(stated, derived)


def to_dev(*ts):
    return [t.cuda() for t in ts]


def run_cuda(shape: ai.AttnShape, q, k, v, workspace=None, with_lse=True):
    import tiled_attention_forward_fwd_gb300 as attn

    o, lse = attn.flash_attn_forward(q.cuda(), k.cuda(), v.cuda(), causal=shape.causal, window=shape.window,
                                     sm_scale=shape.scale, return_lse=with_lse, workspace=workspace)
    st = attn.device_status()
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    return o, lse


def check_full(shape: ai.AttnShape, q, k, v, o_gpu, lse_gpu, oracle_mod, label="", config=None, strict=False):
    kw = dict(causal=shape.causal, window=shape.window, sm_scale=shape.scale)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, **kw)
    a_ref, _ = oracle_mod.attention(q, k, v.abs(), **kw)  # sum_j w_j |V_jc|
    return compare(shape.dtype, o_gpu.float().cpu().numpy(), o_ref,
                   None if lse_gpu is None else lse_gpu.cpu().numpy(), lse_ref, label, a_ref, config, strict)


# Every comparison of the run, for the report printed at the end of the
# session (tests/conftest.py): error against the stated bound, the elements
# over it with their oracle value, and the distance in ulps to the oracle
# rounded to the output dtype.
RECORDS: list[dict] = []
MAX_LISTED = 16  # elements over the stated bound listed per comparison


def ulps_to_rounded(dtype: str, o: np.ndarray, o_ref: np.ndarray) -> float:
    """max |O_gpu - round_dtype(O_oracle)| in ulps of the output grid at the
    rounded oracle value, over the elements with |O_oracle| >= 1/16 (where the
    16-bit grid, not the absolute bound, is what limits the error; 0 when
    there are none): 0 where the kernel returned the correctly rounded
    result."""
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    r = torch.from_numpy(np.ascontiguousarray(o_ref)).to(tdt).to(torch.float64).numpy()
    big = np.abs(o_ref) >= 0.0625
    if not big.any():
        return 0.0
    return float((np.abs(o - r)[big] / dtype_ulp(dtype, r[big])).max())


def compare(dtype, o, o_ref, lse, lse_ref, label="", a_ref=None, config=None, strict=False):
    """Element-by-element check of O and LSE against the oracle.  The O bound
    is the stated one (``strict``) or max(stated, derived) (o_tolerance)."""
    o = o.astype(np.float64)
    assert np.isfinite(o).all(), f"{label}: non-finite output"
    err = np.abs(o - o_ref)
    tol = np.full_like(o_ref, TOL_O[dtype]) if strict else o_tolerance(dtype, o_ref, a_ref)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    over = np.flatnonzero(err.reshape(-1) > TOL_O[dtype])
    order = over[np.argsort(-err.reshape(-1)[over])][:MAX_LISTED]
    stats = {"max_abs_O": float(err.max()), "stated_tol_O": TOL_O[dtype],
             "n_over_stated": int(over.size), "n_elems": int(err.size),
             "O_ref_at_worst": float(o_ref[worst]), "ulps_to_rounded_oracle": ulps_to_rounded(dtype, o, o_ref),
             "over_stated": [(int(i), float(err.reshape(-1)[i]), float(abs(o_ref.reshape(-1)[i]))) for i in order],
             "bound": "stated" if strict else "max(stated, derived)"}
    if lse is not None:
        lerr = np.abs(lse.astype(np.float64) - lse_ref)
        stats["max_abs_LSE"] = float(lerr.max())
    RECORDS.append({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "label": label,
                    "config": config, "dtype": dtype, **stats})
    assert (err <= tol).all(), f"{label}: O error {err[worst]:.3e} > tol {tol[worst]:.3e} at {worst}, " \
                               f"|O_ref|={abs(o_ref[worst]):.3f}; stats {stats}"
    if lse is not None:
        assert stats["max_abs_LSE"] <= TOL_LSE, f"{label}: LSE error {stats['max_abs_LSE']:.3e}"
    return stats


def sample_row_ids(B: int, Hq: int, Nq: int, count: int, seed: int) -> np.ndarray:
    """Stratified query rows: first/last rows, 128-row tile boundaries and
    random rows, spread over random (b, h)."""
    rng = np.random.default_rng(seed)
    special = {0, 1, Nq - 1, Nq - 2}
    for t in range(128, Nq, 128 * max(1, Nq // (128 * 16))):
        special.update({t - 1, t})
    special = sorted(i for i in special if 0 <= i < Nq)
    ids = []
    for i in special:
        ids.append((int(rng.integers(B)) * Hq + int(rng.integers(Hq))) * Nq + i)
    while len(ids) < count:
        ids.append((int(rng.integers(B)) * Hq + int(rng.integers(Hq))) * Nq + int(rng.integers(Nq)))
    return np.unique(np.array(ids[:max(count, len(special))], dtype=np.int64))


def check_sampled(shape: ai.AttnShape, q, k, v, o_gpu, lse_gpu, oracle_mod, count=512, seed=0, label="",
                  config=None, strict=False):
    ids = sample_row_ids(shape.B, shape.Hq, shape.Nq, count, seed)
    d = shape.d
    tid = torch.from_numpy(ids)
    q_rows = q.reshape(-1, d)[tid]
    kw = dict(B=shape.B, Hq=shape.Hq, Nq=shape.Nq, causal=shape.causal, window=shape.window,
              sm_scale=shape.scale)
    o_ref, lse_ref = oracle_mod.attention_rows(q_rows, ids, k, v, **kw)
    a_ref, _ = oracle_mod.attention_rows(q_rows, ids, k, v.abs(), **kw)  # sum_j w_j |V_jc|
    o = o_gpu.reshape(-1, d)[tid.to(o_gpu.device)].float().cpu().numpy()
    lse = None if lse_gpu is None else lse_gpu.reshape(-1)[tid.to(lse_gpu.device)].cpu().numpy()
    return compare(shape.dtype, o, o_ref, lse, lse_ref, label, a_ref, config, strict)


def check_properties(shape, v, o_gpu, lse_gpu):
    """Properties that hold at any size: finite outputs; each O row is a convex
    combination of V rows, so |O| <= max|V| (plus output rounding)."""
    assert torch.isfinite(o_gpu).all()
    vmax = v.abs().max().item()
    assert o_gpu.abs().max().item() <= vmax * (1 + 2 ** -7) + 1e-3
    if lse_gpu is not None:
        assert torch.isfinite(lse_gpu).all()


def scale_of(d):
    return 1.0 / math.sqrt(d)
