"""CPU check of the backward parity bound (tests/test_bwd_gpu.py): the
kernel's arithmetic, emulated in numpy -- P from the fp32 LSE and rounded to
the input dtype, D from the 16-bit O, dS rounded to the input dtype, fp32
scores, 16-bit outputs -- stays within the bound against the fp64 oracle, and
the bound stays a small fraction of the gradient's scale (it is not
vacuous).  A planted mistake in the emulation (dS not multiplied by P)
exceeds it."""
import numpy as np
import pytest
import torch

import attn_inputs as ai
from tests.test_bwd_gpu import bwd_bounds, half_ulp

CASES = [ai.AttnShape(1, 2, 2, 96, 96, 64, "fp16", True), ai.AttnShape(1, 4, 2, 80, 160, 64, "bf16", True),
         ai.AttnShape(1, 2, 1, 64, 64, 64, "bf16", False), ai.AttnShape(1, 2, 2, 100, 100, 64, "fp16", True, 17)]


def r16(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float16 if dtype == "fp16" else torch.bfloat16)
    return t.double().numpy()


def emulate(s, q, k, v, do, oracle_mod, planted=False):
    Q, K, V, G = (t.double().numpy() for t in (q, k, v, do))
    o_ref, lse = oracle_mod.attention(q, k, v, causal=s.causal, window=s.window, sm_scale=s.scale)
    O16 = r16(o_ref, s.dtype)
    g = s.Hq // s.Hkv
    dq, dk, dv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    pos = (s.Nk - s.Nq) + np.arange(s.Nq)[:, None]
    j = np.arange(s.Nk)[None, :]
    live = np.ones((s.Nq, s.Nk), bool)
    if s.causal:
        live &= j <= pos
        if s.window > 0:
            live &= pos - j < s.window
    l2e = np.float32(np.log2(np.e))
    for b in range(s.B):
        for h in range(s.Hq):
            kv = h // g
            S = (s.scale * Q[b, h] @ K[b, kv].T).astype(np.float32)
            P = np.where(live, np.exp2(S * l2e - (lse[b, h][:, None] * l2e).astype(np.float32)), 0.0)
            dP = (G[b, h] @ V[b, kv].T).astype(np.float32)
            D = (G[b, h] * O16[b, h]).sum(axis=1, keepdims=True).astype(np.float32)
            dS = (dP - D) if planted else P * (dP - D)
            P16, dS16 = r16(P, s.dtype), r16(dS, s.dtype)
            dv[b, kv] += P16.T @ G[b, h]
            dk[b, kv] += dS16.T @ Q[b, h]
            dq[b, h] += dS16 @ K[b, kv]
    return (r16(dq * s.scale, s.dtype), r16(dk * s.scale, s.dtype), r16(dv, s.dtype)), O16


def worst_ratio(s, oracle_mod, planted=False):
    q, k, v = ai.make_qkv(s, config_id=161, layer=s.Nq)
    do = ai.normal_tensor(ai.seed_for(161, s.Nq, "G"), tuple(q.shape), s.dtype)
    got, O16 = emulate(s, q, k, v, do, oracle_mod, planted)
    refs = oracle_mod.attention_bwd(q, k, v, do, causal=s.causal, window=s.window, sm_scale=s.scale)
    bnds = bwd_bounds(s, q, k, v, do, torch.from_numpy(O16))
    worst, scale = 0.0, 0.0
    for e, ref, bnd in zip(got, refs, bnds):
        tol = bnd + half_ulp(s.dtype, np.abs(ref) + bnd) + 1e-5 * (np.abs(ref) + bnd) + 1e-6
        worst = max(worst, float(np.max(np.abs(e - ref) / tol)))
        scale = max(scale, float(tol.max() / max(np.abs(ref).max(), 1e-30)))
    return worst, scale


@pytest.mark.parametrize("s", CASES)
def test_emulated_kernel_within_bound(oracle_mod, s):
    worst, scale = worst_ratio(s, oracle_mod)
    assert worst <= 1.0, worst
    assert scale <= 0.05, scale


def test_planted_mistake_exceeds_bound(oracle_mod):
    worst, _ = worst_ratio(CASES[0], oracle_mod, planted=True)
    assert worst > 1.0
