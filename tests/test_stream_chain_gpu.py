"""Calls that depend on each other, back to back on one stream with no host
synchronisation, eagerly and inside a CUDA graph.  Every kernel of the
library is launched with programmatic serialization, so it may start before
the previous kernel on the stream has finished; it must wait
(griddepcontrol.wait) before reading its inputs or writing its outputs.
These tests feed one call's output to the next call (read after write) and
let a call overwrite a buffer the previous call read (write after read)."""
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


def _inputs(shape, cid):
    return [t.cuda() for t in ai.make_qkv(shape, config_id=cid)]


def _chain(attn, graph: bool):
    """prefill (N=2048) -> its O is the query of a short-key call (Nk=64) ->
    that O's last rows are the queries of a split-KV decode call; a fourth
    call writes its O over the first call's Q (read by call 1)."""
    s1 = ai.AttnShape(2, 4, 4, 2048, 2048, 64, "fp16", True)
    q1, k1, v1 = _inputs(s1, 95)
    s2 = ai.AttnShape(2, 4, 2, 2048, 64, 64, "fp16", False)
    _, k2, v2 = _inputs(s2, 96)
    s3 = ai.AttnShape(2, 4, 1, 1, 3000, 64, "fp16", True)
    _, k3, v3 = _inputs(s3, 97)
    o1 = torch.empty_like(q1)
    o2 = torch.empty_like(q1)
    q3 = torch.empty((2, 4, 1, 64), dtype=q1.dtype, device="cuda")
    o3 = torch.empty_like(q3)
    q1_saved = q1.clone()
    o4_into_q1 = q1  # call 4 overwrites call 1's query buffer
    ws = torch.empty(attn.attn_fwd_workspace_bytes(2, 4, 1, 1, 3000, 64), dtype=torch.uint8, device="cuda")
    lse = [torch.empty(t, dtype=torch.float32, device="cuda") for t in ((2, 4, 2048), (2, 4, 2048), (2, 4, 1), (2, 4, 2048))]

    def run():
        attn.flash_attn_forward(q1, k1, v1, causal=True, out=o1, lse=lse[0])
        attn.flash_attn_forward(o1, k2, v2, causal=False, out=o2, lse=lse[1])
        q3.copy_(o2[:, :, -1:, :])
        attn.flash_attn_forward(q3, k3, v3, causal=True, out=o3, lse=lse[2], workspace=ws)
        attn.flash_attn_forward(o2, k1, v1, causal=True, out=o4_into_q1, lse=lse[3])

    assert attn.attn_fwd_path(2, 4, 4, 2048, 2048, 64, False) == attn.ATTN_PATH_PREFILL
    assert attn.attn_fwd_path(2, 4, 2, 2048, 64, 64, False) == attn.ATTN_PATH_SHORT
    assert attn.attn_fwd_path(2, 4, 1, 1, 3000, 64, True) in (attn.ATTN_PATH_SPLIT_KV, attn.ATTN_PATH_SPLIT_KV_FUSED)
    if graph:
        run()  # warm the launch path before capture
        torch.cuda.synchronize()
        q1.copy_(q1_saved)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        q1.copy_(q1_saved)
        torch.cuda.synchronize()
        g.replay()
    else:
        run()
    torch.cuda.synchronize()
    assert attn.device_status() == attn.ATTN_OK
    return (s1, s2, s3), (q1_saved, k1, v1, k2, v2, k3, v3), (o1, o2, q3, o3, o4_into_q1), lse


@pytest.mark.parametrize("graph", [False, True])
def test_dependent_calls_back_to_back(attn, oracle_mod, graph):
    (s1, s2, s3), (q1, k1, v1, k2, v2, k3, v3), (o1, o2, q3, o3, o4), lse = _chain(attn, graph)
    cpu = lambda t: t.cpu()
    # each call against the oracle on the inputs it was given (the previous
    # call's GPU output where it read one)
    pu.check_sampled(s1, cpu(q1), cpu(k1), cpu(v1), o1, lse[0], oracle_mod, count=256, label="call 1")
    pu.check_sampled(s2, cpu(o1), cpu(k2), cpu(v2), o2, lse[1], oracle_mod, count=256, label="call 2 (Q = O1)")
    assert torch.equal(q3, o2[:, :, -1:, :])
    pu.check_full(s3, cpu(q3), cpu(k3), cpu(v3), o3, lse[2], oracle_mod, "call 3 (Q = last rows of O2)")
    s4 = ai.AttnShape(2, 4, 4, 2048, 2048, 64, "fp16", True)
    pu.check_sampled(s4, cpu(o2), cpu(k1), cpu(v1), o4, lse[3], oracle_mod, count=256, label="call 4 (writes over Q1)")


def test_graph_and_eager_chains_agree(attn):
    _, _, outs_e, _ = _chain(attn, False)
    outs_e = [t.clone() for t in outs_e]
    _, _, outs_g, _ = _chain(attn, True)
    for a, b in zip(outs_e, outs_g):
        assert torch.equal(a, b)
