"""GPU parity of the paged prefill (attn_fwd_paged with query groups of more
than 32 rows: the tiled tcgen05 kernel whose TMA producer follows the page
table), through the C ABI, against the fp64 paged oracle.

The motivation page's "PagedAttention es un problema distinto" section: K/V
live in fixed-size pages, each request has a page table and its own length,
and the attention kernel follows the table.  Here the queries are many rows
per request (a prefill, or a chunk of one, against a cache that already
holds earlier tokens): row i of request b sits at position seq_lens[b] - Nq
+ i.  Inputs come from attn_inputs.make_paged: drawn lengths, a shuffled
pool, and NaN in every slot no request owns, so that a read of one shows in
O.  Cases: every page size from 8 to 256 at both head dims, causal and not,
windows, lengths ending inside a page and inside a 128-key tile, the item
shapes of the kernel, bit-identity with the flat call at full length,
device-side length checks, and a CUDA-graph replay with new lengths."""
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


def run(attn, shape, q, k, v, table, lens):
    dev = torch.device("cuda:0")
    s = shape
    assert attn.attn_fwd_paged_path(s.B, s.Hq, s.Hkv, s.Nq, s.max_seq_len, s.d) == attn.ATTN_PATH_PREFILL
    assert attn.attn_fwd_paged_workspace_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.max_seq_len, s.d) == 0
    qd, kd, vd, td, ld = (t.to(dev) for t in (q, k, v, table, lens))
    o, lse = attn.flash_attn_paged(qd, kd, vd, td, ld, s.max_seq_len, s.causal, s.window, s.scale)
    torch.cuda.synchronize()
    return o, lse


def check(attn, oracle_mod, shape, cid, layer=0):
    q, k, v, table, lens = ai.make_paged(shape, cid, layer)
    o, lse = run(attn, shape, q, k, v, table, lens)
    assert attn.device_status() == attn.ATTN_OK
    kw = dict(causal=shape.causal, window=shape.window, sm_scale=shape.scale)
    o_ref, lse_ref = oracle_mod.attention_paged(q, k, v, table, lens, **kw)
    a_ref, _ = oracle_mod.attention_paged(q, k, v.abs(), table, lens, **kw)
    pu.compare(shape.dtype, o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, str(shape), a_ref)
    return q, k, v, table, lens, o, lse


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
@pytest.mark.parametrize("causal", [True, False])
def test_page_sizes_ragged(attn, oracle_mod, page_size, d, dtype, causal):
    """Three requests of drawn lengths (at least the 200 query rows), a
    fragmented pool, NaN in unowned slots."""
    shape = ai.PagedShape(3, 4, 2, 200, 900, d, page_size, dtype, causal, 0, None, None, 200, 3)
    check(attn, oracle_mod, shape, 140, page_size + d + int(causal))


@pytest.mark.parametrize("lens", [(200, 201, 255), (256, 257, 383), (384, 511, 512), (129, 130, 300)])
@pytest.mark.parametrize("page_size", [16, 128])
def test_lengths_at_page_and_tile_edges(attn, oracle_mod, lens, page_size):
    shape = ai.PagedShape(3, 8, 2, 129, 512, 128, page_size, "bf16", True, 0, None, lens, 1, 1)
    check(attn, oracle_mod, shape, 141, sum(lens) + page_size)


@pytest.mark.parametrize("window", [1, 37, 128, 300, 1000])
def test_window(attn, oracle_mod, window):
    shape = ai.PagedShape(2, 4, 4, 300, 1000, 64, 16, "fp16", True, window, None, (1000, 450), 1, 2)
    check(attn, oracle_mod, shape, 142, window)


@pytest.mark.parametrize("Hq,Hkv,Nq,max_len", [
    (8, 4, 1024, 1024),   # two heads of a group per item, full prefill
    (3, 3, 700, 1500),    # odd group: row pairs (chunked prefill, Nq < length)
    (2, 1, 256, 2000),    # few tiles: one tile per item, its K/V tiles split between the warpgroups
    (6, 2, 40, 3000),     # 120-row groups of short chunks
])
def test_item_shapes(attn, oracle_mod, Hq, Hkv, Nq, max_len):
    shape = ai.PagedShape(2, Hq, Hkv, Nq, max_len, 128, 32, "bf16", True, 0, None, None, Nq, 1)
    check(attn, oracle_mod, shape, 143, Hq * 10 + Hkv)


@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
def test_matches_flat_cache_bitwise(attn, d, dtype):
    """With every request at the full length, the paged prefill computes the
    same tiles in the same order as the flat call on the gathered cache:
    identical bits."""
    B, Hq, Hkv, N, ps = 2, 8, 4, 1000, 16
    shape = ai.PagedShape(B, Hq, Hkv, N, N, d, ps, dtype, True, 0, None, (N,) * B, 1, 0)
    q, k, v, table, lens = ai.make_paged(shape, 144, d)
    o, lse = run(attn, shape, q, k, v, table, lens)
    assert attn.device_status() == attn.ATTN_OK
    pages = -(-N // ps)
    idx = table[:, :pages].long()
    kf = k[idx].permute(0, 2, 1, 3, 4).reshape(B, Hkv, pages * ps, d)[:, :, :N].contiguous()
    vf = v[idx].permute(0, 2, 1, 3, 4).reshape(B, Hkv, pages * ps, d)[:, :, :N].contiguous()
    flat = ai.AttnShape(B, Hq, Hkv, N, N, d, dtype, True)
    of, lf = pu.run_cuda(flat, q, kf, vf)
    assert torch.equal(o.cpu(), of.cpu())
    assert torch.equal(lse.cpu(), lf.cpu())


def test_bad_length_reported(attn):
    """A length below the query rows (causal) is found on the device,
    clamped, and reported as ATTN_ERR_DEVICE_ARG; the call finishes."""
    shape = ai.PagedShape(2, 4, 2, 100, 400, 64, 16, "fp16", True, 0, None, (400, 300), 1, 0)
    q, k, v, table, lens = ai.make_paged(shape, 145, 0)
    bad = lens.clone()
    bad[1] = 50
    run(attn, shape, q, k, v, table, bad)
    assert attn.device_status() == attn.ATTN_ERR_DEVICE_ARG
    assert attn.device_status() == attn.ATTN_OK


def test_graph_replay_with_new_lengths(attn, oracle_mod):
    """A captured prefill over a paged cache replays with new queries and
    lengths written in place (the lengths are read on the device)."""
    max_len = 1500
    shape = ai.PagedShape(2, 8, 2, 300, max_len, 128, 64, "bf16", True, 0, None, (max_len, max_len), 1, 1)
    q, k, v, table, lens = ai.make_paged(shape, 146, 0)
    dev = torch.device("cuda:0")
    qd, kd, vd, td, ld = (t.to(dev) for t in (q, k, v, table, lens))
    o = torch.empty_like(qd)
    lse = torch.empty((2, 8, 300), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        attn.flash_attn_paged(qd, kd, vd, td, ld, max_len, out=o, lse=lse)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            attn.flash_attn_paged(qd, kd, vd, td, ld, max_len, out=o, lse=lse)
    torch.cuda.synchronize()
    for r, new in enumerate([(1500, 300), (301, 1499), (1000, 1000)], start=1):
        qn = ai.normal_tensor(ai.seed_for(146, r, "Q"), tuple(q.shape), "bf16")
        qd.copy_(qn)
        nl = torch.tensor(new, dtype=torch.int32)
        ld.copy_(nl)
        g.replay()
        torch.cuda.synchronize()
        assert attn.device_status() == attn.ATTN_OK
        o_ref, lse_ref = oracle_mod.attention_paged(qn, k, v, table, nl, True)
        pu.compare("bf16", o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, f"replay {r} {new}")


def test_workload_sampled(attn, oracle_mod):
    """The benchmark's chunked prefill at full size (4 requests, 2048 new rows
    each, caches of drawn lengths up to 8192): per request, sampled rows
    against the oracle on the request's cache gathered from its pages."""
    s, cid, layer = ai.workload_calls("paged_prefill")[0]
    q, k, v, table, lens = ai.make_paged(s, cid, layer)
    o, lse = run(attn, s, q, k, v, table, lens)
    assert attn.device_status() == attn.ATTN_OK
    ps = s.page_size
    for b in range(s.B):
        n = int(lens[b])
        pages = table[b, :(n + ps - 1) // ps].long()
        kf = k[pages].permute(1, 0, 2, 3).reshape(s.Hkv, -1, s.d)[:, :n][None].contiguous()
        vf = v[pages].permute(1, 0, 2, 3).reshape(s.Hkv, -1, s.d)[:, :n][None].contiguous()
        flat = ai.AttnShape(1, s.Hq, s.Hkv, s.Nq, n, s.d, s.dtype, s.causal, s.window, s.sm_scale)
        pu.check_sampled(flat, q[b:b + 1], kf, vf, o[b:b + 1], lse[b:b + 1], oracle_mod, count=192, seed=b,
                         label=f"paged_prefill[{b}]",
                         config=f"C-paged paged_prefill request {b} of 4 Hq32 Hkv8 Nq2048 L{n} ps16 d128 causal")
