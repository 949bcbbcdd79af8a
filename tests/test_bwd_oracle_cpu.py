"""Pins of the backward oracle (oracle.attention_bwd), on CPU.

The gradients are fixed by the forward definition, so they are checked
against things other than their own formula:

* central finite differences of the forward oracle (pinned on its own in
  test_oracle_pins.py), element by element on tiny inputs and along random
  directions on larger ones;
* torch float64 autograd of softmax(Q K^T * scale + mask) V (a library
  routine; GQA as repeat_interleave of K and V);
* closed forms: with all keys equal, the weights do not depend on Q (dQ = 0)
  and dV_j is the sum of dO_i / |J(i)| over the rows that see key j;
* invariants: shifting every key by one vector leaves O unchanged, so the
  key gradients of a head sum to zero under any mask; the gradients are
  linear in dO.
"""
import math

import numpy as np
import pytest
import torch

import oracle

TIGHT = 1e-12


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def loss(q, k, v, do, causal, window, scale):
    o, _ = oracle.attention(q, k, v, causal, window, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal,window,Hq,Hkv", [(False, 0, 2, 1), (True, 0, 2, 2), (True, 2, 4, 2)])
def test_finite_differences_elementwise(causal, window, Hq, Hkv):
    B, N, d, scale, h = 1, 5, 3, 0.7, 1e-5
    q, k, v, do = rnd((B, Hq, N, d), 1), rnd((B, Hkv, N, d), 2), rnd((B, Hkv, N, d), 3), rnd((B, Hq, N, d), 4)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, window, scale)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = loss(*[xp if n == name else args[n] for n in "qkv"], do, causal, window, scale)
            lm = loss(*[xm if n == name else args[n] for n in "qkv"], do, causal, window, scale)
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 9)])
def test_finite_differences_directional(causal, window):
    """Nq < Nk (bottom-right causal), GQA 6/2, along random directions."""
    B, Hq, Hkv, Nq, Nk, d, scale, h = 2, 6, 2, 11, 23, 8, 0.4, 1e-5
    q, do = rnd((B, Hq, Nq, d), 11), rnd((B, Hq, Nq, d), 14)
    k, v = rnd((B, Hkv, Nk, d), 12), rnd((B, Hkv, Nk, d), 13)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, window, scale)
    for seed, (name, g) in enumerate((("q", dq), ("k", dk), ("v", dv))):
        base = {"q": q, "k": k, "v": v}
        u = rnd(base[name].shape, 100 + seed)
        plus = dict(base, **{name: base[name] + h * u})
        minus = dict(base, **{name: base[name] - h * u})
        num = (loss(plus["q"], plus["k"], plus["v"], do, causal, window, scale) -
               loss(minus["q"], minus["k"], minus["v"], do, causal, window, scale)) / (2 * h)
        assert abs(float(np.sum(g * u)) - num) <= 1e-7 * max(1.0, abs(num)), name


@pytest.mark.parametrize("causal,window,Hq,Hkv,Nq,Nk", [(False, 0, 4, 4, 40, 40), (True, 0, 4, 1, 40, 40),
                                                         (True, 7, 6, 2, 30, 50), (False, 0, 2, 1, 1, 64)])
def test_torch_autograd(causal, window, Hq, Hkv, Nq, Nk):
    B, d, scale = 2, 16, 0.25
    q, k, v, do = rnd((B, Hq, Nq, d), 21), rnd((B, Hkv, Nk, d), 22), rnd((B, Hkv, Nk, d), 23), rnd((B, Hq, Nq, d), 24)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    g = Hq // Hkv
    kk, vv = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
    s = tq @ kk.transpose(-1, -2) * scale
    pos = torch.arange(Nq)[:, None] + (Nk - Nq)
    j = torch.arange(Nk)[None, :]
    keep = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:
        keep &= j <= pos
        if window > 0:
            keep &= pos - j < window
    s = s.masked_fill(~keep, float("-inf"))
    (torch.softmax(s, dim=-1) @ vv).backward(torch.tensor(do))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, window, scale)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=TIGHT)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=TIGHT)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=TIGHT)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 4)])
def test_identical_keys(causal, window):
    B, Hq, Hkv, N, d = 1, 4, 2, 13, 5
    q, v, do = rnd((B, Hq, N, d), 31), rnd((B, Hkv, N, d), 32), rnd((B, Hq, N, d), 33)
    k = np.broadcast_to(rnd((d,), 34), (B, Hkv, N, d)).copy()
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, window, 0.5)
    assert np.abs(dq).max() < TIGHT
    want = np.zeros_like(v)
    for h in range(Hq):
        for i in range(N):
            live = [j for j in range(N) if (not causal or j <= i) and (window <= 0 or i - j < window)]
            for j in live:
                want[0, h // (Hq // Hkv), j] += do[0, h, i] / len(live)
    np.testing.assert_allclose(dv, want, rtol=0, atol=TIGHT)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3)])
def test_key_shift_invariance(causal, window):
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 9, 17, 6
    q, k, v, do = rnd((B, Hq, Nq, d), 41), rnd((B, Hkv, Nk, d), 42), rnd((B, Hkv, Nk, d), 43), rnd((B, Hq, Nq, d), 44)
    _, dk, _ = oracle.attention_bwd(q, k, v, do, causal, window, 0.6)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12
    # and the gradients at shifted keys are the same
    dq0, dk0, dv0 = oracle.attention_bwd(q, k, v, do, causal, window, 0.6)
    dq1, dk1, dv1 = oracle.attention_bwd(q, k + rnd((d,), 45), v, do, causal, window, 0.6)
    for a, b in ((dq0, dq1), (dk0, dk1), (dv0, dv1)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_linear_in_do():
    B, Hq, Hkv, N, d = 1, 2, 1, 12, 4
    q, k, v = rnd((B, Hq, N, d), 51), rnd((B, Hkv, N, d), 52), rnd((B, Hkv, N, d), 53)
    a, b = rnd((B, Hq, N, d), 54), rnd((B, Hq, N, d), 55)
    ga = oracle.attention_bwd(q, k, v, a, True)
    gb = oracle.attention_bwd(q, k, v, b, True)
    gab = oracle.attention_bwd(q, k, v, 2 * a - b, True)
    for x, y, z in zip(ga, gb, gab):
        np.testing.assert_allclose(z, 2 * x - y, rtol=0, atol=TIGHT)


def test_rows_without_keys_rejected():
    q = rnd((1, 1, 5, 4), 61)
    k = rnd((1, 1, 3, 4), 62)
    with pytest.raises(ValueError):
        oracle.attention_bwd(q, k, k, q, True)  # causal with Nq > Nk: rows 0, 1 see no key
    assert math.isfinite(oracle.attention_bwd(q, k, k, q, False)[0].sum())
