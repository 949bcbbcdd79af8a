"""The host-buffer entry (attn_fwd_host) on the GPU: copies in, the call, and
copies out, enqueued on one stream.

Large calls are cut into pieces of (request, K/V head) slabs whose copies
overlap the compute of their neighbours (include/attn.h, attn_fwd_host).
Each piece runs with the whole call's schedule, so the output must be the
same bits as the device-buffer call (attn_fwd_ex) on the same inputs, whether
or not the call is cut; the device-buffer call's parity with the oracle is
checked elsewhere, and once here on sampled rows."""
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


def host_call(attn, s, qh, kh, vh, with_lse=True, stream=None):
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32).pin_memory() if with_lse else None
    need = attn.attn_fwd_host_staging_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, with_lse)
    buf = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    base = (buf.data_ptr() + 255) & ~255
    stream = stream or torch.cuda.current_stream()
    st = attn.attn_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                            lh.data_ptr() if with_lse else None, s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, s.causal,
                            s.window, s.scale, attn.ATTN_DTYPE_BF16 if s.dtype == "bf16" else attn.ATTN_DTYPE_FP16,
                            base, need, stream.cuda_stream)
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    stream.synchronize()
    assert attn.device_status() == attn.ATTN_OK
    return oh, lh, buf


def device_call(attn, s, q, k, v):
    nb = attn.attn_fwd_workspace_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None
    return pu.run_cuda(s, q, k, v, workspace=ws)


CASES = [
    # cut into 8 pieces of one K/V head (B = 1, GQA 32 / 8, 100 MB of inputs)
    ai.AttnShape(1, 32, 8, 8192, 8192, 128, "bf16", True),
    # cut into 8 pieces of one request (B = 8, 16 / 4 heads, d = 64, non-causal)
    ai.AttnShape(8, 16, 4, 4096, 4096, 64, "fp16", False),
    # windowed, cut by K/V heads of two requests
    ai.AttnShape(2, 16, 4, 8192, 8192, 128, "bf16", True, 1000),
    # a smaller call: not cut (copy, compute, copy on the stream)
    ai.AttnShape(2, 4, 4, 1024, 1024, 64, "fp16", True),
    # MHA with an odd group: pieces would pair tiles differently, so not cut
    ai.AttnShape(8, 12, 12, 2048, 2048, 64, "bf16", True, 0, 0.125),
]


@pytest.mark.parametrize("s", CASES, ids=[f"B{c.B}_H{c.Hq}/{c.Hkv}_N{c.Nq}_d{c.d}_c{int(c.causal)}_w{c.window}"
                                          for c in CASES])
def test_same_bits_as_device_call(attn, oracle_mod, s):
    q, k, v = ai.make_qkv(s, config_id=180)
    o_dev, l_dev = device_call(attn, s, q, k, v)
    oh, lh, _ = host_call(attn, s, q.pin_memory(), k.pin_memory(), v.pin_memory())
    assert torch.equal(oh, o_dev.cpu())
    assert torch.equal(lh, l_dev.cpu())
    pu.check_sampled(s, q, k, v, oh, lh, oracle_mod, count=128, seed=3, label="host path")


def test_without_lse_and_on_a_side_stream(attn):
    s = CASES[0]
    q, k, v = ai.make_qkv(s, config_id=181)
    o_dev, _ = device_call(attn, s, q, k, v)
    side = torch.cuda.Stream()
    oh, _, _ = host_call(attn, s, q.pin_memory(), k.pin_memory(), v.pin_memory(), with_lse=False, stream=side)
    assert torch.equal(oh, o_dev.cpu())


def test_graph_capture_replays_with_new_inputs(attn):
    """A call large enough to be cut, captured in a CUDA graph (under
    capture it runs uncut on the stream), replayed after the pinned inputs
    change in place; meanwhile an eager call on another stream is cut and
    stays out of the graph."""
    s = CASES[0]
    q, k, v = ai.make_qkv(s, config_id=182)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32).pin_memory()
    need = attn.attn_fwd_host_staging_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, True)
    buf = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    base = (buf.data_ptr() + 255) & ~255
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st = attn.attn_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), lh.data_ptr(), s.B, s.Hq,
                                s.Hkv, s.Nq, s.Nk, s.d, s.causal, s.window, s.scale, attn.ATTN_DTYPE_BF16, base, need,
                                torch.cuda.current_stream().cuda_stream)
        assert st == attn.ATTN_OK
    # an eager (cut) call while the graph exists: it must not touch the graph's buffers
    q3, k3, v3 = ai.make_qkv(s, config_id=189)
    o3, _, _ = host_call(attn, s, q3.pin_memory(), k3.pin_memory(), v3.pin_memory())
    o3_dev, _ = device_call(attn, s, q3, k3, v3)
    assert torch.equal(o3, o3_dev.cpu())
    for rep in range(3):
        q2, k2, v2 = ai.make_qkv(s, config_id=183 + rep)
        qh.copy_(q2)
        kh.copy_(k2)
        vh.copy_(v2)
        g.replay()
        torch.cuda.synchronize()
        o_dev, l_dev = device_call(attn, s, q2, k2, v2)
        assert torch.equal(oh, o_dev.cpu()), rep
        assert torch.equal(lh, l_dev.cpu()), rep
    assert attn.device_status() == attn.ATTN_OK
