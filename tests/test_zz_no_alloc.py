"""The decode entry point that allocates nothing (attn_fwd_decode_noalloc).

Some callers cannot give the library any device memory: their device memory
is owned entirely by their own pool with no hook for plugins, or they may not
call cudaMalloc while work is in flight.  This entry point serves them with
the split-KV decode running on a scratch block built into the library.  The
tests call it through the C ABI and compare it with the regular entry point
(attn_fwd_ex with a caller workspace) on two calls in a row, so the second
call runs on the scratch contents the first one left behind.

The file name makes pytest collect it last."""
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


def call_noalloc(attn, shape, q, k, v):
    o = torch.empty_like(q)
    lse = torch.empty((shape.B, shape.Hq, shape.Nq), device=q.device, dtype=torch.float32)
    code = attn.ATTN_DTYPE_BF16 if shape.dtype == "bf16" else attn.ATTN_DTYPE_FP16
    st = attn.attn_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d, shape.causal,
                                      shape.window, shape.scale, code,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    assert attn.device_status() == attn.ATTN_OK
    return o, lse


def call_with_workspace(attn, shape, q, k, v):
    nbytes = attn.attn_fwd_workspace_bytes(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    return attn.flash_attn_forward(q, k, v, causal=shape.causal, window=shape.window, sm_scale=shape.scale,
                                   workspace=ws)


def test_two_calls_match_the_workspace_entry(attn, oracle_mod):
    # the decode workload (MQA, then GQA with 8 K/V heads): two calls in a
    # row, each also checked element by element against the fp64 oracle
    for idx in range(2):
        shape, cid, layer = ai.workload_calls("mqa_decode")[idx]
        qh, kh, vh = ai.make_qkv(shape, config_id=cid, layer=layer)
        q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
        o_ref, lse_ref = call_with_workspace(attn, shape, q, k, v)
        o, lse = call_noalloc(attn, shape, q, k, v)
        assert (o.float() - o_ref.float()).abs().max().item() <= pu.TOL_O[shape.dtype]
        assert (lse - lse_ref).abs().max().item() <= pu.TOL_LSE
        pu.check_full(shape, qh, kh, vh, o, lse, oracle_mod, f"no-alloc decode, call {idx + 1}")


def test_second_call_with_other_inputs(attn):
    """A smaller shape after a larger one: stale scratch must not leak in."""
    for cid, shape in [(70, ai.AttnShape(2, 16, 2, 2, 3000, 64, "fp16", True, 700)),
                       (71, ai.AttnShape(1, 8, 8, 4, 257, 128, "bf16", False))]:
        q, k, v = (t.cuda() for t in ai.make_qkv(shape, config_id=cid))
        o_ref, lse_ref = call_with_workspace(attn, shape, q, k, v)
        o, lse = call_noalloc(attn, shape, q, k, v)
        assert (o.float() - o_ref.float()).abs().max().item() <= pu.TOL_O[shape.dtype]
        assert (lse - lse_ref).abs().max().item() <= pu.TOL_LSE


def test_rejects_what_does_not_fit(attn):
    # 64 query rows per K/V head: this shape does not take the split-KV path
    q = torch.zeros(1, 8, 64, 64, device="cuda", dtype=torch.float16)
    kv = torch.zeros(1, 8, 512, 64, device="cuda", dtype=torch.float16)
    o = torch.empty_like(q)
    st = attn.attn_fwd_decode_noalloc(q.data_ptr(), kv.data_ptr(), kv.data_ptr(), o.data_ptr(), None, 1, 8, 8, 64,
                                      512, 64, 1, 0, 0.125, attn.ATTN_DTYPE_FP16,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_SCRATCH_LIMIT
    # a decode shape whose scratch exceeds the built-in 8 MiB: 16384 query rows, one key chunk each
    B, Hq, Nk, d = 512, 32, 64, 128
    big = attn.attn_fwd_workspace_bytes(B, Hq, 1, 1, Nk, d)
    assert big > 8 << 20
    qb = torch.zeros(B, Hq, 1, d, device="cuda", dtype=torch.bfloat16)
    kb = torch.zeros(B, 1, Nk, d, device="cuda", dtype=torch.bfloat16)
    ob = torch.empty_like(qb)
    st = attn.attn_fwd_decode_noalloc(qb.data_ptr(), kb.data_ptr(), kb.data_ptr(), ob.data_ptr(), None, B, Hq, 1,
                                      1, Nk, d, 1, 0, 0.088, attn.ATTN_DTYPE_BF16,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_ERR_SCRATCH_LIMIT
    assert attn.device_status() == attn.ATTN_OK
