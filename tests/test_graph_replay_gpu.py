"""Split paths replayed from a CUDA graph with new inputs written in place.

The split-KV decode (cruxr.ai "FlashDecoding": chunks of the keys processed
in parallel, then merged) and the d = 128 prefill split both combine partial
results that different CTAs of one launch wrote to the workspace.  A CTA must
merge the partials of its own launch: a graph replays the launch parameters
it captured, so nothing taken on the host at enqueue time can tell one
replay's partials from the previous replay's.  Each case captures one call,
then replays it several times, rewriting Q, K and V (and, for a paged cache,
the request lengths) in place before every replay, and compares every replay
with the oracle on the inputs of that replay.  Where the workspace still held
the previous replay's partials, a merge that did not wait for its own would
show as a mismatch."""
import pytest
import torch

import attn_inputs as ai
from tests import parity_util as pu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

REPLAYS = 6


@pytest.fixture(scope="module")
def attn():
    import tiled_attention_forward_fwd_gb300 as m

    m.lib()
    return m


def capture(fn):
    """Warm the launch path, then capture fn() into a graph on a side stream."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


FLAT_CASES = [
    # (shape, expected path); decode steps whose merge is fused (one launch)
    # or done by the merge kernel, and two d = 128 prefills that take the
    # stream-K split
    (ai.AttnShape(2, 4, 4, 1, 3000, 128, "bf16", True), "fused"),
    (ai.AttnShape(2, 4, 2, 1, 5000, 64, "fp16", True, 1000), "fused"),  # window: the early chunks are empty
    (ai.AttnShape(1, 32, 1, 1, 4096, 128, "bf16", True), "merge kernel"),
    (ai.AttnShape(1, 4, 4, 700, 700, 128, "bf16", True), "prefill split"),
    (ai.AttnShape(1, 8, 2, 1100, 1500, 128, "bf16", False), "prefill split"),
]


def expected_path(attn, kind):
    return {"fused": attn.ATTN_PATH_SPLIT_KV_FUSED, "merge kernel": attn.ATTN_PATH_SPLIT_KV,
            "prefill split": attn.ATTN_PATH_PREFILL_SPLIT}[kind]


@pytest.mark.parametrize("shape,kind", FLAT_CASES, ids=[f"{k}-{i}" for i, (_, k) in enumerate(FLAT_CASES)])
def test_flat_split_replays(attn, oracle_mod, shape, kind):
    s = shape
    assert attn.attn_fwd_path(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, True) == expected_path(attn, kind)
    q, k, v = (t.cuda() for t in ai.make_qkv(s, config_id=120, layer=0))
    ws = torch.empty(attn.attn_fwd_workspace_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0xA5)  # garbage in the workspace before the first call, handshake words included
    o = torch.empty_like(q)
    lse = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32, device="cuda")
    g = capture(lambda: attn.flash_attn_forward(q, k, v, causal=s.causal, window=s.window, sm_scale=s.scale,
                                                out=o, lse=lse, workspace=ws))
    for r in range(1, REPLAYS + 1):
        qh, kh, vh = ai.make_qkv(s, config_id=120, layer=r)
        q.copy_(qh)
        k.copy_(kh)
        v.copy_(vh)
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert attn.device_status() == attn.ATTN_OK
        pu.check_full(s, qh, kh, vh, o, lse, oracle_mod, f"{kind} replay {r}")
    # an eager call on the same workspace after the replays
    qh, kh, vh = ai.make_qkv(s, config_id=120, layer=REPLAYS + 1)
    q.copy_(qh)
    k.copy_(kh)
    v.copy_(vh)
    attn.flash_attn_forward(q, k, v, causal=s.causal, window=s.window, sm_scale=s.scale, out=o, lse=lse,
                            workspace=ws)
    torch.cuda.synchronize()
    pu.check_full(s, qh, kh, vh, o, lse, oracle_mod, f"{kind} eager after replays")


@pytest.mark.parametrize("Hq,Hkv,d,kind", [(4, 4, 128, "fused"), (8, 8, 64, "fused"), (16, 4, 128, "merge kernel")])
def test_paged_replays_with_new_lengths(attn, oracle_mod, Hq, Hkv, d, kind):
    """A decode loop on a paged cache: each replay sees new queries and new
    request lengths.  The pages are allocated for the longest length; some
    replays leave the later key chunks of a request empty, others fill them."""
    max_len, ps = 5000, 16
    shape = ai.PagedShape(3, Hq, Hkv, 1, max_len, d, ps, "bf16", True, 0, None, (max_len,) * 3, 1, 2)
    assert attn.attn_fwd_paged_path(3, Hq, Hkv, 1, max_len, d) == expected_path(attn, kind)
    q, k, v, table, lens = ai.make_paged(shape, 121, 0)
    qd, kd, vd, td, ld = (t.cuda() for t in (q, k, v, table, lens))
    ws = torch.empty(attn.attn_fwd_paged_workspace_bytes(3, Hq, Hkv, 1, max_len, d), dtype=torch.uint8,
                     device="cuda")
    ws.fill_(0x5A)
    o = torch.empty_like(qd)
    lse = torch.empty((3, Hq, 1), dtype=torch.float32, device="cuda")
    g = capture(lambda: attn.flash_attn_paged(qd, kd, vd, td, ld, max_len, out=o, lse=lse, workspace=ws))
    steps = [(5000, 17, 2049), (64, 4999, 2048), (1, 1, 1), (3000, 5000, 4097), (5000, 5000, 5000),
             (129, 2500, 4096)]
    assert len(steps) == REPLAYS
    for r, new_lens in enumerate(steps, start=1):
        qn = ai.normal_tensor(ai.seed_for(121, r, "Q"), tuple(q.shape), "bf16")
        qd.copy_(qn)
        nl = torch.tensor(new_lens, dtype=torch.int32)
        ld.copy_(nl)
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert attn.device_status() == attn.ATTN_OK
        o_ref, lse_ref = oracle_mod.attention_paged(qn, k, v, table, nl, True)
        pu.compare("bf16", o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, f"paged replay {r} {new_lens}")


@pytest.mark.parametrize("d", [64, 128])
def test_backward_replays(attn, d):
    """The backward (a pre-pass that zeroes the dQ accumulator, the kernel that
    reduce-adds every key tile's dQ part into it, then the dQ pass) captured
    once and replayed with a new dO written in place each time: every replay
    equals an eager call on the same inputs (the accumulator starts from
    zero in every replay), up to the order in which the CTAs' fp32
    reduce-adds land."""
    s = ai.AttnShape(2, 4, 2, 600, 600, d, "bf16", True)
    q, k, v = (t.cuda() for t in ai.make_qkv(s, config_id=195))
    o, lse = attn.flash_attn_forward(q, k, v, causal=True)
    do = torch.empty_like(q)
    ws = torch.empty(attn.attn_bwd_workspace_bytes(s.B, s.Hq, s.Nq, s.d), dtype=torch.uint8, device="cuda")
    out = {}

    def call():
        out["g"] = attn.flash_attn_backward(q, k, v, o, lse, do, True, workspace=ws)

    do.copy_(ai.normal_tensor(ai.seed_for(195, 0, "G"), tuple(q.shape), s.dtype).cuda())
    g = capture(call)
    for r in range(REPLAYS):
        do.copy_(ai.normal_tensor(ai.seed_for(195, r + 1, "G"), tuple(q.shape), s.dtype).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert attn.device_status() == attn.ATTN_OK
        got = [t.clone() for t in out["g"]]
        want = attn.flash_attn_backward(q, k, v, o, lse, do, True)
        torch.cuda.synchronize()
        for name, a, b in zip(("dQ", "dK", "dV"), got, want):
            assert torch.isfinite(a.float()).all(), (r, name)
            # the reduce-adds of different CTAs may land in another order
            # in the two launches (fp32 sums): compare within the rounding
            # of a few fp32 additions on top of the 16-bit output
            torch.testing.assert_close(a.float(), b.float(), rtol=2e-2, atol=2e-3, msg=f"replay {r} {name}")
