"""GPU parity of decode over an INT8 K/V cache (attn_fwd_kv_int8, through the
C ABI) against the fp64 oracle on the same codes and scales.

cruxr.ai "Optimizaciones de Atencion", section "Elegir optimizaciones de
atencion": INT8 quantisation of the KV cache composes with the other
optimisations.  The scheme (reading R17): symmetric codes in [-127, 127], one
fp32 scale per tensor, K = k_scale * codes, V = v_scale * codes.  The kernel
loads the codes, widens them exactly to the dtype of Q and folds the scales
into the softmax scale and into O; the oracle dequantises exactly in fp64 and
runs the plain definition (oracle.attention_kv_int8, pinned on CPU).  The
tolerance is the same as for 16-bit K/V, with |V| = v_scale * |codes|."""
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


def check(attn, oracle_mod, shape, cid, layer=0, config=None, path=None):
    s = shape
    q, kc, ks, vc, vs = ai.make_qkv_int8(s, cid, layer)
    if path is not None:
        assert attn.attn_fwd_path(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, True) == getattr(attn, path)
    o, lse = attn.flash_attn_kv_int8(q.cuda(), kc.cuda(), vc.cuda(), ks, vs, s.causal, s.window, s.scale)
    assert attn.device_status() == attn.ATTN_OK
    kw = dict(causal=s.causal, window=s.window, sm_scale=s.scale)
    o_ref, lse_ref = oracle_mod.attention_kv_int8(q, kc, vc, ks, vs, **kw)
    a_ref, _ = oracle_mod.attention_kv_int8(q, kc, vc.abs(), ks, vs, **kw)  # sum_j w_j |V_jc|
    return pu.compare(s.dtype, o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, str(s), a_ref, config)


@pytest.mark.parametrize("idx", [0, 1])
def test_workload(attn, oracle_mod, idx):
    """The benchmark's int8 decode step (mqa_decode's shapes), every row."""
    shape, cid, layer = ai.workload_calls("mqa_decode_int8")[idx]
    check(attn, oracle_mod, shape, cid, layer,
          config=f"C-dec mqa_decode_int8 B4 Hq32 Hkv{shape.Hkv} Nq1 Nk8192 d128 causal int8 K/V")


@pytest.mark.parametrize("Nk", [1, 2, 63, 64, 65, 129, 1000, 5000])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16"), (128, "fp16"), (64, "bf16")])
def test_ragged_keys(attn, oracle_mod, Nk, d, dtype):
    shape = ai.AttnShape(2, 8, 2, 1, Nk, d, dtype, True, kv_int8=True)
    check(attn, oracle_mod, shape, 150, Nk + d)


@pytest.mark.parametrize("B,Hq,Hkv,Nq", [(1, 32, 1, 1), (2, 8, 2, 4), (3, 4, 4, 7), (2, 2, 1, 16), (1, 1, 1, 32)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300)])
def test_groups_and_queries(attn, oracle_mod, B, Hq, Hkv, Nq, causal, window):
    shape = ai.AttnShape(B, Hq, Hkv, Nq, 1500, 128, "bf16", causal, window, kv_int8=True)
    check(attn, oracle_mod, shape, 151, Hq * 100 + Nq)


@pytest.mark.parametrize("shape,path", [
    (ai.AttnShape(2, 4, 4, 1, 3000, 128, "bf16", True, kv_int8=True), "ATTN_PATH_SPLIT_KV_FUSED"),
    (ai.AttnShape(1, 32, 1, 1, 4096, 128, "fp16", True, kv_int8=True), "ATTN_PATH_SPLIT_KV"),
    (ai.AttnShape(2, 4, 2, 1, 5000, 64, "fp16", True, 1000, kv_int8=True), "ATTN_PATH_SPLIT_KV_FUSED"),
])
def test_both_merges(attn, oracle_mod, shape, path):
    check(attn, oracle_mod, shape, 152, shape.Nk, path=path)


def test_scaled_keys_stress(attn, oracle_mod):
    """Keys x3 before quantisation (peaked softmax rows, the long-context
    workload's stress): the key scale folded into the softmax scale."""
    shape = ai.AttnShape(2, 16, 2, 2, 4000, 128, "bf16", True, key_scale=3.0, kv_int8=True)
    check(attn, oracle_mod, shape, 153)


def test_errors(attn):
    dev = "cuda"
    q = torch.zeros(1, 8, 1, 128, device=dev, dtype=torch.bfloat16)
    kc = torch.zeros(1, 2, 300, 128, device=dev, dtype=torch.int8)
    for ks, vs in [(0.0, 1.0), (1.0, float("nan")), (-1.0, 1.0)]:
        with pytest.raises(attn.AttnError) as e:
            attn.flash_attn_kv_int8(q, kc, kc, ks, vs)
        assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    big = torch.zeros(1, 8, 64, 128, device=dev, dtype=torch.bfloat16)  # 256 rows per K/V head
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_kv_int8(big, kc, kc, 1.0, 1.0, causal=False)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED
    assert attn.device_status() == attn.ATTN_OK
