"""The parity tolerance, checked on the CPU against a simulation of the
arithmetic the pages prescribe: exact fp64 scores and weights, probabilities
rounded to the value dtype before P V (lab 02: ``p.to(v.dtype)``), O divided
by the fp32-style unrounded sum and stored in the value dtype.  The derived
bound must hold for that simulation, and the simulation must show that the
stated max-abs bound alone cannot always be met (so the derived term is
needed, not a loosening)."""
import math

import numpy as np
import pytest
import torch

from attn_inputs import normal_tensor
from tests import parity_util as pu

DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def simulate(q, k, v, dtype, causal, window, scale):
    """Per row: p_j = exp(s_j - max) rounded to dtype; O = sum p~ V / sum p."""
    q, k, v = (x.to(torch.float64) for x in (q, k, v))
    N = q.shape[2]
    S = (q @ k.transpose(-1, -2)) * scale
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    keep = torch.ones(N, N, dtype=torch.bool)
    if causal:
        keep &= j <= i
    if window > 0:
        keep &= (i - j) < window
    S = S.masked_fill(~keep, float("-inf"))
    p = torch.exp(S - S.amax(-1, keepdim=True))
    pr = p.to(DT[dtype]).to(torch.float64)
    o = (pr @ v) / p.sum(-1, keepdim=True)
    return o.to(DT[dtype]).to(torch.float64).numpy()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 2), (True, 5)])
def test_derived_bound_covers_exact_arithmetic(oracle_mod, dtype, causal, window):
    N, d = 96, 32
    worst_over_stated = 0.0
    for seed in range(3):
        q = normal_tensor(500 + seed, (1, 2, N, d), dtype)
        k = normal_tensor(600 + seed, (1, 2, N, d), dtype, scale=3.0)
        v = normal_tensor(700 + seed, (1, 2, N, d), dtype, scale=1.5)
        scale = 1 / math.sqrt(d)
        o_ref, _ = oracle_mod.attention(q, k, v, causal=causal, window=window, sm_scale=scale)
        a_ref, _ = oracle_mod.attention(q, k, v.abs(), causal=causal, window=window, sm_scale=scale)
        o_sim = simulate(q, k, v, dtype, causal, window, scale)
        err = np.abs(o_sim - o_ref)
        tol = pu.o_tolerance(dtype, o_ref, a_ref)
        assert (err <= tol).all(), (err - tol).max()
        worst_over_stated = max(worst_over_stated, err.max() / pu.TOL_O[dtype])
    # record: whether the pages' own arithmetic exceeds the stated bound here
    print(dtype, causal, window, "max err / stated bound:", round(worst_over_stated, 3))


def test_stated_bound_alone_is_not_attainable(oracle_mod):
    """bf16, two live keys per row, large |V|: the exact arithmetic of the
    pages already exceeds 8e-3, so the derived term is required."""
    N, d = 64, 16
    q = normal_tensor(11, (1, 1, N, d), "bf16")
    k = normal_tensor(12, (1, 1, N, d), "bf16", scale=0.2)
    v = normal_tensor(13, (1, 1, N, d), "bf16", scale=3.0)
    o_ref, _ = oracle_mod.attention(q, k, v, causal=True, window=2, sm_scale=0.25)
    o_sim = simulate(q, k, v, "bf16", True, 2, 0.25)
    assert np.abs(o_sim - o_ref).max() > pu.TOL_O["bf16"]
