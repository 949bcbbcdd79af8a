"""GPU parity of the short-key path (Nk <= 128: one tile of keys per head,
softmax over the whole row), through the C ABI, against the fp64 oracle."""
import pytest
import torch

import attn_inputs as ai
from tests import parity_util as pu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def attn():
    import tiled_attention_forward_fwd_gb300 as m

    m.lib()
    return m


def _check(shape, oracle_mod, cid, layer=0):
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"{shape}")


@pytest.mark.parametrize("Nk", [1, 2, 33, 64, 65, 100, 128])
@pytest.mark.parametrize("Nq", [1, 7, 64, 65, 130])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
def test_short_keys_non_causal(attn, oracle_mod, Nk, Nq, d, dtype):
    """Both key-tile widths (64 / 128 rows, zero-filled past Nk), query
    blocks of 64 rows with a ragged last block."""
    _check(ai.AttnShape(2, 3, 3, Nq, Nk, d, dtype, False), oracle_mod, 70, Nk * 1000 + Nq)


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 128), (5, 40), (40, 40), (64, 64), (63, 128), (100, 128),
                                   (128, 128)])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "fp16")])
def test_short_keys_causal(attn, oracle_mod, Nq, Nk, d, dtype):
    """Bottom-right causal alignment with Nq <= Nk."""
    _check(ai.AttnShape(2, 2, 1, Nq, Nk, d, dtype, True), oracle_mod, 71, Nk * 1000 + Nq)


@pytest.mark.parametrize("window", [1, 2, 17, 64, 127])
def test_short_keys_window(attn, oracle_mod, window):
    _check(ai.AttnShape(1, 4, 2, 90, 128, 64, "fp16", True, window), oracle_mod, 72, window)


@pytest.mark.parametrize("Hkv", [1, 2, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_short_keys_gqa(attn, oracle_mod, Hkv, d):
    _check(ai.AttnShape(2, 8, Hkv, 70, 96, d, "bf16", True), oracle_mod, 73, Hkv)


def test_many_units_per_cta(attn, oracle_mod):
    """More units than resident CTAs: the persistent loop wraps the ring."""
    _check(ai.AttnShape(64, 16, 16, 64, 64, 64, "fp16", True), oracle_mod, 74)


@pytest.mark.parametrize("idx", [0, 1])
def test_mha_n64_bandwidth_full_size(attn, oracle_mod, idx):
    """B=512, H=32, N=64, d=64 fp16 (the bandwidth-sized N=64 workload):
    sampled rows against the oracle, properties everywhere."""
    shape, cid, layer = ai.workload_calls("mha_n64_bw")[idx]
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_properties(shape, v.cuda(), o, lse)
    pu.check_sampled(shape, q, k, v, o, lse, oracle_mod, count=1024, label="mha_n64_bw",
                     config=f"C1-bw mha_n64_bw B512 H32 N64 d64{' causal' if shape.causal else ''} (1024 rows)",
                     strict=True)
