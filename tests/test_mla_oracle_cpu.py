"""Pins of the latent-cache (MLA) oracle, oracle.attention_mla, on CPU.

cruxr.ai "Optimizaciones de Atencion", "Multi-Head Latent Attention (MLA)":
the cache holds one latent vector per token, keys and values are rebuilt by
up-projections, and the same attention can be computed without rebuilding
them by absorbing the up-projections into the query and output sides.  The
oracle rebuilds K and V explicitly; these tests pin it with:

* the absorbed form, computed independently with torch in float64: per head
  q~ = W_K,h^up q (length d_c), scores q~ . c_t, a softmax over the shared
  latent keys, o~ = sum_t p_t c_t, then O = o~ W_V,h^up -- the mathematics
  is the same, the arithmetic path is not;
* a special case that reduces to plain MHA: with d_c = n_h * d_h and
  identity up-projections the latent is the keys (and values) of all heads
  side by side.
"""
import numpy as np
import pytest
import torch

import oracle


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def absorbed(q, c, wk, wv, causal, window, scale):
    q, c, wk, wv = (torch.tensor(x) for x in (q, c, wk, wv))
    B, n_h, Nq, d_h = q.shape
    Nk, d_c = c.shape[1], c.shape[2]
    wk_h = wk.reshape(d_c, n_h, d_h)  # W_K,h^up = wk_h[:, h, :]
    wv_h = wv.reshape(d_c, n_h, d_h)
    q_lat = torch.einsum("bhid,chd->bhic", q, wk_h)  # absorbed queries, length d_c
    s = torch.einsum("bhic,btc->bhit", q_lat, c) * scale
    pos = torch.arange(Nq)[:, None] + (Nk - Nq)
    t = torch.arange(Nk)[None, :]
    keep = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:
        keep &= t <= pos
        if window > 0:
            keep &= pos - t < window
    s = s.masked_fill(~keep, float("-inf"))
    p = torch.softmax(s, dim=-1)
    o_lat = torch.einsum("bhit,btc->bhic", p, c)  # weighted latent, length d_c
    o = torch.einsum("bhic,chd->bhid", o_lat, wv_h)
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("causal,window,Nq", [(False, 0, 1), (True, 0, 1), (True, 0, 4), (True, 5, 3)])
def test_absorbed_form(causal, window, Nq):
    B, n_h, d_h, d_c, Nk = 2, 4, 16, 32, 40
    q = rnd((B, n_h, Nq, d_h), 1)
    c = rnd((B, Nk, d_c), 2)
    wk, wv = rnd((d_c, n_h * d_h), 3, 0.2), rnd((d_c, n_h * d_h), 4, 0.2)
    o, lse = oracle.attention_mla(q, c, wk, wv, causal, window)
    oa, la = absorbed(q, c, wk, wv, causal, window, 1.0 / np.sqrt(d_h))
    np.testing.assert_allclose(o, oa, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, la, rtol=0, atol=1e-12)


def test_identity_projection_is_mha():
    B, n_h, d_h, Nk, Nq = 2, 3, 8, 25, 25
    d_c = n_h * d_h
    q = rnd((B, n_h, Nq, d_h), 11)
    c = rnd((B, Nk, d_c), 12)
    eye = np.eye(d_c)
    o, lse = oracle.attention_mla(q, c, eye, eye, True)
    kv = c.reshape(B, Nk, n_h, d_h).transpose(0, 2, 1, 3)  # head h = latent columns [h*d_h, (h+1)*d_h)
    om, lm = oracle.attention(q, kv, kv, causal=True)
    np.testing.assert_array_equal(o, om)
    np.testing.assert_array_equal(lse, lm)


def test_shapes_rejected():
    with pytest.raises(ValueError):
        oracle.attention_mla(np.zeros((1, 2, 1, 4)), np.zeros((1, 5, 8)), np.zeros((8, 7)), np.zeros((8, 7)))
