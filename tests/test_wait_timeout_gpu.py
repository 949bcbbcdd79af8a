"""Bounded waits that run out, on the GPU.

Every wait inside the kernels (an mbarrier of the TMA ring or of the
tensor-core handoffs, a flag of the prefill split) gives up after a limit
(attn_set_wait_timeout_ns; 2 s by default), records ATTN_ERR_TIMEOUT in the
device status word, and the CTA winds down: every role skips its remaining
copies and MMAs but keeps its fixed sequence of barriers, the producers wait
for the copies they issued, and TMEM is freed.

Two ways in.  (1) A limit of 1 ns: any wait that polls more than once runs
out (how many do depends on timing).  (2) The test hook
attn_set_test_stall(k): every producer stops loading after k K/V tiles, so
the roles waiting for the next tile wait on something that never comes and
run into their limit (here 200 us) -- a timeout, deterministically, in the
middle of the pipeline.  Each call must come back, the status must read as
expected, and with the hooks off the next call on the same buffers must
match the oracle again."""
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
    yield m
    m.attn_set_wait_timeout_ns(0)  # default limit
    m.attn_set_test_stall(-1)


CASES = [
    # (shape, with workspace, path)
    (ai.AttnShape(1, 2, 2, 300, 300, 64, "fp16", False), False, "ATTN_PATH_PREFILL"),
    (ai.AttnShape(2, 4, 2, 700, 900, 128, "bf16", True), False, "ATTN_PATH_PREFILL"),
    (ai.AttnShape(1, 2, 2, 1000, 1000, 64, "bf16", False), False, "ATTN_PATH_PREFILL"),  # halves items
    (ai.AttnShape(1, 4, 4, 700, 700, 128, "bf16", True), True, "ATTN_PATH_PREFILL_SPLIT"),
    (ai.AttnShape(2, 4, 4, 1, 3000, 128, "bf16", True), True, "ATTN_PATH_SPLIT_KV_FUSED"),
    (ai.AttnShape(1, 32, 1, 1, 4096, 128, "bf16", True), True, "ATTN_PATH_SPLIT_KV"),
    (ai.AttnShape(2, 4, 4, 200, 100, 64, "fp16", False), False, "ATTN_PATH_SHORT"),
]
IDS = [c[2] + f"-{i}" for i, c in enumerate(CASES)]


def _setup(attn, shape, with_ws, path):
    s = shape
    assert attn.attn_fwd_path(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, with_ws) == getattr(attn, path)
    q, k, v = ai.make_qkv(s, config_id=130)
    ws = None
    if with_ws:
        ws = torch.zeros(attn.attn_fwd_workspace_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d), dtype=torch.uint8,
                         device="cuda")
    o = torch.empty((s.B, s.Hq, s.Nq, s.d), dtype=q.dtype, device="cuda")
    lse = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32, device="cuda")
    return (q, k, v), (q.cuda(), k.cuda(), v.cuda()), ws, o, lse


def _call(attn, s, dev, ws, o, lse):
    qd, kd, vd = dev
    attn.flash_attn_forward(qd, kd, vd, causal=s.causal, window=s.window, sm_scale=s.scale, out=o, lse=lse,
                            workspace=ws)
    return attn.device_status()  # synchronises: the call came back


def _recovered(attn, oracle_mod, s, host, dev, ws, o, lse, label):
    attn.attn_set_wait_timeout_ns(0)
    attn.attn_set_test_stall(-1)
    if ws is not None:
        ws.zero_()  # a launch that timed out may leave a handshake word set
    assert _call(attn, s, dev, ws, o, lse) == attn.ATTN_OK
    q, k, v = host
    pu.check_full(s, q, k, v, o, lse, oracle_mod, label)


@pytest.mark.parametrize("shape,with_ws,path", CASES, ids=IDS)
def test_tiny_limit_then_recovery(attn, oracle_mod, shape, with_ws, path):
    host, dev, ws, o, lse = _setup(attn, shape, with_ws, path)
    assert attn.device_status() == attn.ATTN_OK
    try:
        attn.attn_set_wait_timeout_ns(1)
        for _ in range(3):
            st = _call(attn, shape, dev, ws, o, lse)
            assert st in (attn.ATTN_OK, attn.ATTN_ERR_TIMEOUT), attn.attn_status_string(st)
    finally:
        attn.attn_set_wait_timeout_ns(0)
    _recovered(attn, oracle_mod, shape, host, dev, ws, o, lse, f"{path} after a 1 ns limit")


# (case, tiles loaded before the stall): below the tile count of the CTAs,
# so that they stall (here the short-key kernel's CTAs hold one unit each, the
# merge-kernel decode's chunks one tile, and the prefill split gives each CTA
# one K/V step)
ONE_TILE = ("ATTN_PATH_SHORT", "ATTN_PATH_SPLIT_KV", "ATTN_PATH_PREFILL_SPLIT")
STALLS = [(i, k) for i in range(len(CASES)) for k in ((0,) if CASES[i][2] in ONE_TILE else (0, 1))] + \
    [(0, 2), (2, 3)]


@pytest.mark.parametrize("case,stall", STALLS, ids=[f"{IDS[i]}-stall{k}" for i, k in STALLS])
def test_stalled_producer_times_out(attn, oracle_mod, case, stall):
    shape, with_ws, path = CASES[case]
    host, dev, ws, o, lse = _setup(attn, shape, with_ws, path)
    assert attn.device_status() == attn.ATTN_OK
    try:
        attn.attn_set_wait_timeout_ns(200_000)
        attn.attn_set_test_stall(stall)
        st = _call(attn, shape, dev, ws, o, lse)
        assert st == attn.ATTN_ERR_TIMEOUT, attn.attn_status_string(st)
        assert attn.device_status() == attn.ATTN_OK  # read and cleared
    finally:
        attn.attn_set_wait_timeout_ns(0)
        attn.attn_set_test_stall(-1)
    _recovered(attn, oracle_mod, shape, host, dev, ws, o, lse, f"{path} after a stall at tile {stall}")
