"""Pins of the INT8 K/V-cache oracle (oracle.attention_kv_int8), on CPU.

With symmetric per-tensor codes, K = s_k * codes_K and V = s_v * codes_V, so
(i) the key scale can be folded into the softmax scale, and (ii) the value
scale multiplies O and leaves LSE alone; the oracle dequantises first
instead.  These identities, computed through the plain (pinned) oracle on
the raw codes, pin it; so does the trivial scale of 1.  The quantiser that
makes test inputs (attn_inputs.quantize_int8) is checked on its own: codes
within [-127, 127], round-trip error at most half a step."""
import numpy as np
import pytest
import torch

import attn_inputs as ai
import oracle


def rnd(shape, seed):
    return torch.from_numpy(np.random.default_rng(seed).standard_normal(shape))


@pytest.mark.parametrize("causal,window,Hq,Hkv,Nq,Nk", [(False, 0, 4, 4, 30, 30), (True, 0, 8, 2, 1, 70),
                                                         (True, 6, 4, 1, 12, 40)])
def test_scale_folding(causal, window, Hq, Hkv, Nq, Nk):
    B, d, scale = 2, 16, 0.3
    q = rnd((B, Hq, Nq, d), 1)
    kc, sk = ai.quantize_int8(rnd((B, Hkv, Nk, d), 2) * 2.5)
    vc, sv = ai.quantize_int8(rnd((B, Hkv, Nk, d), 3))
    o, lse = oracle.attention_kv_int8(q, kc, vc, sk, sv, causal, window, scale)
    # keys: the code attention with the key scale folded into sm_scale; values: O times v_scale
    o_codes, lse_codes = oracle.attention(q, kc.double(), vc.double(), causal=causal, window=window,
                                          sm_scale=scale * sk)
    np.testing.assert_allclose(o, sv * o_codes, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_codes, rtol=0, atol=1e-12)


def test_unit_scales_are_plain_attention():
    q = rnd((1, 2, 9, 8), 11)
    kc = torch.randint(-127, 128, (1, 2, 9, 8), generator=torch.Generator().manual_seed(0), dtype=torch.int8)
    vc = torch.randint(-127, 128, (1, 2, 9, 8), generator=torch.Generator().manual_seed(1), dtype=torch.int8)
    o, lse = oracle.attention_kv_int8(q, kc, vc, 1.0, 1.0, True, 0, 0.01)
    o2, lse2 = oracle.attention(q, kc.double(), vc.double(), causal=True, sm_scale=0.01)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_quantizer():
    x = rnd((3, 4, 50, 16), 21) * 3.0
    codes, s = ai.quantize_int8(x.to(torch.bfloat16))
    assert codes.dtype == torch.int8 and int(codes.abs().max()) <= 127 and int(codes.abs().max()) >= 126
    err = (codes.double() * s - x.to(torch.bfloat16).double()).abs().max().item()
    assert err <= s / 2 * (1 + 1e-6)


def test_bad_codes_rejected():
    q = rnd((1, 1, 2, 4), 31)
    with pytest.raises(ValueError):
        oracle.attention_kv_int8(q, np.full((1, 1, 2, 4), 128.0), np.zeros((1, 1, 2, 4)), 1.0, 1.0)
    with pytest.raises(ValueError):
        oracle.attention_kv_int8(q, np.full((1, 1, 2, 4), 0.5), np.zeros((1, 1, 2, 4)), 1.0, 1.0)
    with pytest.raises(ValueError):
        oracle.attention_kv_int8(q, np.zeros((1, 1, 2, 4)), np.zeros((1, 1, 2, 4)), 0.0, 1.0)
