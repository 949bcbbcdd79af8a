"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle
on the same seeded inputs, element by element."""
import numpy as np
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


def _run_and_check(shape, oracle_mod, config_id=50, layer=0, label="", config=None, strict=False):
    q, k, v = ai.make_qkv(shape, config_id=config_id, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    return pu.check_full(shape, q, k, v, o, lse, oracle_mod, label or str(shape), config, strict)


def _name(workload, shape):
    return (f"{workload} B{shape.B} Hq{shape.Hq} Hkv{shape.Hkv} Nq{shape.Nq} Nk{shape.Nk} d{shape.d}"
            f"{' causal' if shape.causal else ''}{f' w{shape.window}' if shape.window else ''}")


# ------------------------------------------------------------------ the stated workloads (small ones in full)
@pytest.mark.parametrize("idx", [0, 1])
def test_mha_n64(attn, oracle_mod, idx):
    shape, cid, layer = ai.workload_calls("mha_n64")[idx]
    _run_and_check(shape, oracle_mod, cid, layer, config=_name("C1 mha_n64", shape), strict=True)


@pytest.mark.parametrize("idx", range(6))
def test_mha_b2h4(attn, oracle_mod, idx):
    shape, cid, layer = ai.workload_calls("mha_b2h4")[idx]
    _run_and_check(shape, oracle_mod, cid, layer, config=_name("C2 mha_b2h4", shape), strict=True)


# ------------------------------------------------------------------ ragged and tiny shapes
@pytest.mark.parametrize("N", [1, 2, 15, 16, 17, 63, 65, 127, 128, 129, 255, 257, 300])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (64, "bf16"), (128, "fp16"), (128, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged(attn, oracle_mod, N, d, dtype, causal):
    shape = ai.AttnShape(1, 2, 1, N, N, d, dtype, causal)
    _run_and_check(shape, oracle_mod, 51, N)


@pytest.mark.parametrize("Hkv", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_gqa_groups(attn, oracle_mod, Hkv, d):
    shape = ai.AttnShape(2, 8, Hkv, 300, 300, d, "bf16", True)
    _run_and_check(shape, oracle_mod, 52, Hkv)


@pytest.mark.parametrize("window", [1, 2, 37, 127, 128, 129, 300, 699, 700, 5000])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
def test_sliding_window(attn, oracle_mod, window, d, dtype):
    shape = ai.AttnShape(1, 4, 2, 700, 700, d, dtype, True, window)
    _run_and_check(shape, oracle_mod, 53, window)


@pytest.mark.parametrize("Nq", [1, 5, 128, 130, 300, 777])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 200)])
def test_queries_fewer_than_keys(attn, oracle_mod, Nq, causal, window):
    """Nq < Nk: bottom-right causal alignment (the queries are the last Nq
    positions); decode is Nq = 1."""
    shape = ai.AttnShape(2, 4, 2, Nq, 777, 128, "fp16", causal, window)
    _run_and_check(shape, oracle_mod, 54, Nq)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("key_scale", [3.0, 8.0])
def test_rescale_stress(attn, oracle_mod, d, key_scale):
    """Scores that grow along the key axis, so the running row maximum rises on
    every K/V tile (exercising the lazy rescale of O), with large magnitudes:
    every query is a fixed direction u plus noise, key j is
    key_scale * (j / N) * u plus noise."""
    N = 1000
    shape = ai.AttnShape(1, 2, 2, N, N, d, "fp16", False)
    u = ai.normal_tensor(80 + d, (d,), "f64")
    noise_q = ai.normal_tensor(81, (1, 2, N, d), "f64") * 0.1
    noise_k = ai.normal_tensor(82, (1, 2, N, d), "f64")
    ramp = torch.arange(N, dtype=torch.float64)[None, None, :, None] / N
    q = (u + noise_q).to(torch.float16)
    k = (key_scale * ramp * u + noise_k).to(torch.float16)
    v = ai.normal_tensor(83, (1, 2, N, d), "fp16")
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, "rescale stress")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("kind,x", [("step", 0.5), ("step", 1.5), ("step", 3.0), ("spike", 7.5)])
def test_rescale_triggers(attn, oracle_mod, dtype, kind, x):
    """Scores set per K/V tile of 128 keys, so that the decision to rescale is
    taken exactly at the lazy-rescale threshold.  "stepX": every key of tile b
    scores b*X (log2 units, row 0); the running sum of a tile then exceeds
    2^8 once the max has grown by more than 1, although the max grows by less
    than 8 per tile.  "spikeX": one key per tile scores b*X, the others far
    below; p reaches 2^7.5 without a rescale on odd tiles and forces one on
    even tiles.  Row i scales every score by 1 + (i % 7) / 7."""
    N, d = 2048, 64
    shape = ai.AttnShape(1, 2, 2, N, N, d, dtype, False)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    ln2 = float(np.log(2.0))
    blk = torch.arange(N, dtype=torch.float64) // 128
    c = blk * x * ln2  # natural-log units; d^-1/2 * q0 = 1 below
    if kind == "spike":
        c = torch.where(torch.arange(N) % 128 == 5, c, torch.full_like(c, -30.0))
    q = torch.zeros(1, 2, N, d, dtype=torch.float64)
    q[..., 0] = 8.0 * (1.0 + (torch.arange(N) % 7) / 7.0)
    k = torch.zeros(1, 2, N, d, dtype=torch.float64)
    k[..., 0] = c
    k[..., 1:] = ai.normal_tensor(84, (1, 2, N, d - 1), "f64") * 0.01
    v = ai.normal_tensor(85, (1, 2, N, d), "f64")
    q, k, v = q.to(tdt), k.to(tdt), v.to(tdt)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"rescale triggers {kind} {x}")


def test_lse_optional_and_streams(attn, oracle_mod):
    shape = ai.AttnShape(2, 4, 4, 333, 333, 64, "fp16", True)
    q, k, v = ai.make_qkv(shape, config_id=56)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = pu.run_cuda(shape, q, k, v, with_lse=False)
    s.synchronize()
    assert lse is None
    o_ref, _ = oracle_mod.attention(q, k, v, causal=True)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= pu.TOL_O["fp16"]


def test_outputs_fully_overwritten(attn, oracle_mod):
    shape = ai.AttnShape(1, 2, 2, 130, 130, 64, "fp16", False)
    q, k, v = ai.make_qkv(shape, config_id=57)
    out = torch.full((1, 2, 130, 64), float("nan"), device="cuda", dtype=torch.float16)
    lse = torch.full((1, 2, 130), float("nan"), device="cuda")
    attn.flash_attn_forward(q.cuda(), k.cuda(), v.cuda(), out=out, lse=lse)
    assert attn.device_status() == attn.ATTN_OK
    pu.check_full(shape, q, k, v, out, lse, oracle_mod)


def test_bad_arguments_return_status(attn):
    q = torch.zeros(1, 3, 64, 64, device="cuda", dtype=torch.float16)
    k = torch.zeros(1, 2, 64, 64, device="cuda", dtype=torch.float16)
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_forward(q, k, k)  # Hq % Hkv != 0
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    q2 = torch.zeros(1, 2, 64, 96, device="cuda", dtype=torch.float16)
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_forward(q2, q2, q2)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED
    q3 = torch.zeros(1, 2, 65, 64, device="cuda", dtype=torch.float16)
    kv = torch.zeros(1, 2, 64, 64, device="cuda", dtype=torch.float16)
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_forward(q3, kv, kv, causal=True)  # causal with Nq > Nk
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_forward(kv, kv, kv, causal=False, window=8)
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    assert attn.device_status() == attn.ATTN_OK


# ------------------------------------------------------------------ full-size workloads, sampled rows
@pytest.mark.parametrize("layer", [0, 11])
def test_gpt_stack_full_size(attn, oracle_mod, layer):
    shape, cid, _ = ai.workload_calls("gpt_stack")[layer]
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_properties(shape, v, o, lse)
    pu.check_sampled(shape, q, k, v, o, lse, oracle_mod, count=512, seed=layer, label=f"gpt layer {layer}",
                     config=_name(f"C3 gpt_stack layer {layer}", shape) + " (512 sampled rows)", strict=True)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_gqa_mqa_full_size(attn, oracle_mod, idx):
    shape, cid, layer = ai.workload_calls("gqa_mqa")[idx]
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_properties(shape, v, o, lse)
    pu.check_sampled(shape, q, k, v, o, lse, oracle_mod, count=512, seed=idx, label=f"gqa_mqa {idx}",
                     config=_name("C4 gqa_mqa", shape) + " (512 sampled rows)", strict=shape.window == 0)


def test_long_prefill_full_size(attn, oracle_mod):
    shape, cid, layer = ai.workload_calls("long_prefill")[0]
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_properties(shape, v, o, lse)
    stats = pu.check_sampled(shape, q, k, v, o, lse, oracle_mod, count=768, seed=4, label="long prefill",
                             config=_name("C5 long_prefill", shape) + " (768 sampled rows)")
    print("long_prefill", stats)
