"""GPU parity of the split-KV (decode / small query count) path, through the
C ABI with a caller workspace, against the fp64 oracle."""
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


def run_split(attn, shape, q, k, v):
    """Run the split-KV kernels: through attn_fwd_ex with a workspace where the
    shape takes that path (Nk > 128), else through attn_fwd_decode_noalloc,
    which always runs them (attn_fwd_ex sends Nk <= 128 to the short-key
    kernel)."""
    nbytes = attn.attn_fwd_workspace_bytes(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d)
    assert nbytes > 0, "shape should qualify for the split-KV path"
    path = attn.attn_fwd_path(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d, True)
    if path in (attn.ATTN_PATH_SPLIT_KV, attn.ATTN_PATH_SPLIT_KV_FUSED):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        return pu.run_cuda(shape, q, k, v, workspace=ws)
    assert path == attn.ATTN_PATH_SHORT and shape.Nk <= 128
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((shape.B, shape.Hq, shape.Nq), device="cuda", dtype=torch.float32)
    code = attn.ATTN_DTYPE_BF16 if shape.dtype == "bf16" else attn.ATTN_DTYPE_FP16
    st = attn.attn_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d, shape.causal,
                                      shape.window, shape.scale, code, torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    assert attn.device_status() == attn.ATTN_OK
    return o, lse


@pytest.mark.parametrize("idx", [0, 1])
def test_mqa_decode_workload(attn, oracle_mod, idx):
    shape, cid, layer = ai.workload_calls("mqa_decode")[idx]
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = run_split(attn, shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"mqa_decode {idx}",
                  config=f"C-dec mqa_decode B4 Hq32 Hkv{shape.Hkv} Nq1 Nk8192 d128 causal", strict=True)


@pytest.mark.parametrize("Nk", [1, 2, 63, 64, 65, 129, 1000, 5000])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16"), (128, "fp16"), (64, "bf16")])
def test_decode_ragged_keys(attn, oracle_mod, Nk, d, dtype):
    shape = ai.AttnShape(2, 8, 2, 1, Nk, d, dtype, True)
    q, k, v = ai.make_qkv(shape, config_id=60, layer=Nk)
    o, lse = run_split(attn, shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod)


@pytest.mark.parametrize("B,Hq,Hkv,Nq", [(1, 32, 1, 1), (2, 8, 2, 4), (3, 4, 4, 7), (1, 16, 1, 2),
                                         (2, 2, 1, 16), (1, 1, 1, 32), (2, 6, 3, 9)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300)])
def test_decode_groups_and_queries(attn, oracle_mod, B, Hq, Hkv, Nq, causal, window):
    """Up to 32 query rows per K/V head (g * Nq), bottom-right causal
    alignment, sliding window."""
    shape = ai.AttnShape(B, Hq, Hkv, Nq, 1500, 128, "bf16", causal, window)
    q, k, v = ai.make_qkv(shape, config_id=61, layer=Hq * 100 + Nq)
    o, lse = run_split(attn, shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod)


def test_decode_matches_prefill_path(attn):
    """The same call with and without a workspace (split-KV vs prefill path)."""
    shape = ai.AttnShape(2, 16, 2, 2, 3000, 128, "fp16", True)
    q, k, v = ai.make_qkv(shape, config_id=62)
    o_s, l_s = run_split(attn, shape, q, k, v)
    o_p, l_p = pu.run_cuda(shape, q, k, v)
    assert (o_s.float() - o_p.float()).abs().max().item() <= 2e-3
    assert (l_s - l_p).abs().max().item() <= 1e-4


def test_workspace_errors_and_fallback(attn):
    shape = ai.AttnShape(1, 32, 1, 1, 512, 128, "bf16", True)
    q, k, v = (t.cuda() for t in ai.make_qkv(shape, config_id=63))
    need = attn.attn_fwd_workspace_bytes(1, 32, 1, 1, 512, 128)
    small = torch.empty(need - 4, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_forward(q, k, v, causal=True, workspace=small)
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    # more than 32 query rows per K/V head: no split-KV; a prefill this small
    # takes the stream-K split instead, with its own size and the same check
    assert attn.attn_fwd_path(1, 32, 1, 2, 512, 128, True) == attn.ATTN_PATH_PREFILL_SPLIT
    need2 = attn.attn_fwd_workspace_bytes(1, 32, 1, 2, 512, 128)
    assert need2 > need
    shape2 = ai.AttnShape(1, 32, 1, 2, 512, 128, "bf16", True)
    q2, k2, v2 = (t.cuda() for t in ai.make_qkv(shape2, config_id=63))
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_forward(q2, k2, v2, causal=True, workspace=torch.empty(need2 - 4, dtype=torch.uint8,
                                                                               device="cuda"))
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    # a prefill with enough tile pairs for two waves takes no workspace, nor
    # does one at d = 64
    assert attn.attn_fwd_workspace_bytes(8, 12, 12, 2048, 2048, 128) == 0
    assert attn.attn_fwd_workspace_bytes(1, 32, 1, 2, 512, 64) == 0
    assert attn.device_status() == attn.ATTN_OK


def test_workspace_reuse_is_stateless(attn, oracle_mod):
    """A workspace holding stale data from another call gives the same result."""
    shape = ai.AttnShape(1, 8, 1, 3, 2000, 64, "fp16", True)
    q, k, v = ai.make_qkv(shape, config_id=64)
    nbytes = attn.attn_fwd_workspace_bytes(1, 8, 1, 3, 2000, 64)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device="cuda")  # garbage floats
    o1, l1 = pu.run_cuda(shape, q, k, v, workspace=ws)
    o2, l2 = pu.run_cuda(shape, q, k, v, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    pu.check_full(shape, q, k, v, o1, l1, oracle_mod)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,ws,expect", [
    (4, 32, 8, 1, 8192, True, 4), (4, 32, 1, 1, 8192, True, 1), (4, 32, 8, 1, 8192, False, 0),
    (4, 32, 8, 1, 128, True, 2),
    (2, 4, 4, 64, 64, False, 2), (2, 4, 4, 256, 256, True, 3), (2, 4, 4, 256, 256, False, 0),
    (1, 32, 1, 2, 4096, True, 3), (1, 4, 4, 33, 4096, True, 3), (4, 32, 8, 8192, 8192, True, 0),
    (8, 12, 12, 2048, 2048, True, 0), (2, 8, 0, 1, 64, False, -1)])
def test_path_selection(attn, B, Hq, Hkv, Nq, Nk, ws, expect):
    """attn_fwd_path (d = 128): short keys first; with a workspace, split-KV
    when the group has at most 32 query rows (its merge fused into the split
    kernel when small: 4 query rows x 9 chunks), else the stream-K prefill split
    when the tile pairs fill less than two waves of SMs; else prefill; -1 on
    bad sizes.  At d = 64 the prefill split is never taken."""
    assert attn.attn_fwd_path(B, Hq, Hkv, Nq, Nk, 128, ws) == expect
    if expect == 3:
        assert attn.attn_fwd_path(B, Hq, Hkv, Nq, Nk, 64, ws) == 0
