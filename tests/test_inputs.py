"""The seeded input generator: published splitmix64 outputs, N(0,1) moments,
determinism, and the key scale applied before the single rounding."""
import numpy as np
import torch

import attn_inputs as ai


def test_splitmix64_published_vector():
    # splitmix64 with state 0 (Vigna's reference splitmix64.c): first outputs
    out = ai.splitmix64(0, 0, 3)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_slices_agree():
    a = ai.splitmix64(1234, 0, 100)
    b = ai.splitmix64(1234, 40, 60)
    assert np.array_equal(a[40:], b)


def test_normal_moments():
    z = ai.normal_f64(7, 1 << 20)
    assert abs(z.mean()) < 5e-3
    assert abs(z.var() - 1.0) < 5e-3
    assert abs((z ** 4).mean() - 3.0) < 0.05  # Gaussian kurtosis
    assert np.isfinite(z).all()


def test_odd_length_and_chunks():
    z = ai.normal_f64(9, 2 * ai._CHUNK + 3)
    z2 = ai.normal_f64(9, 5)
    assert np.array_equal(z[:5], z2)


def test_rounding_once_with_scale():
    z = ai.normal_f64(5, 1000) * 3.0
    t = ai.normal_tensor(5, (1000,), "bf16", scale=3.0)
    assert torch.equal(t, torch.from_numpy(z).to(torch.bfloat16))
    t16 = ai.normal_tensor(5, (10, 100), "fp16")
    assert t16.dtype == torch.float16 and t16.shape == (10, 100)


def test_make_qkv_shapes_and_determinism():
    s = ai.AttnShape(B=2, Hq=4, Hkv=2, Nq=3, Nk=5, d=8, dtype="bf16", key_scale=3.0)
    q, k, v = ai.make_qkv(s, config_id=5)
    assert q.shape == (2, 4, 3, 8) and k.shape == (2, 2, 5, 8) and v.shape == (2, 2, 5, 8)
    q2, k2, v2 = ai.make_qkv(s, config_id=5)
    assert ai.sha256_of(q) == ai.sha256_of(q2) and torch.equal(k, k2) and torch.equal(v, v2)
    assert not torch.equal(ai.make_qkv(s, config_id=6)[0], q)
    assert ai.seed_for(4, 3, "V") == 4032
