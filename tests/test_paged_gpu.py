"""GPU parity of attention over a paged K/V cache (attn_fwd_paged, through the
C ABI) against the fp64 paged oracle.

The motivation page's "PagedAttention es un problema distinto" section: K/V
live in fixed-size pages, each request has a page table and its own length,
and the kernel follows the table.  Inputs come from attn_inputs.make_paged:
per-request lengths, a shuffled (fragmented) pool, and NaN in every slot no
request owns, so that a read of one shows in O.  Cases cover every page size
from 8 to 256, lengths ending inside a page and inside a tile, both merges
of the split-KV kernel, windows, several query rows per request, and the
device-side checks of page indices and lengths."""
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


def run_paged(attn, shape, q, k, v, table, lens, ws_extra=0):
    dev = torch.device("cuda:0")
    qd, kd, vd, td, ld = (t.to(dev) for t in (q, k, v, table, lens))
    need = attn.attn_fwd_paged_workspace_bytes(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.max_seq_len, shape.d)
    assert need > 0
    ws = torch.empty(need + ws_extra, dtype=torch.uint8, device=dev)
    o, lse = attn.flash_attn_paged(qd, kd, vd, td, ld, shape.max_seq_len, shape.causal, shape.window, shape.scale,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.ATTN_OK
    return o, lse


def check(attn, oracle_mod, shape, cid, layer=0, config=None, strict=False):
    q, k, v, table, lens = ai.make_paged(shape, cid, layer)
    o, lse = run_paged(attn, shape, q, k, v, table, lens)
    kw = dict(causal=shape.causal, window=shape.window, sm_scale=shape.scale)
    o_ref, lse_ref = oracle_mod.attention_paged(q, k, v, table, lens, **kw)
    a_ref, _ = oracle_mod.attention_paged(q, k, v.abs(), table, lens, **kw)
    pu.compare(shape.dtype, o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, str(shape), a_ref, config,
               strict)
    return q, k, v, table, lens, o, lse


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("d", [64, 128])
def test_page_sizes_ragged(attn, oracle_mod, page_size, d):
    """Eight requests of drawn lengths (1..3000) over a shuffled pool."""
    shape = ai.PagedShape(8, 16, 2, 1, 3000, d, page_size, "bf16", True, 0, None, None, 1, 7)
    check(attn, oracle_mod, shape, 100, page_size + d)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq", [1, 3])
def test_lengths_inside_pages_and_tiles(attn, oracle_mod, dtype, causal, Nq):
    """Lengths at, just past and just short of page (16) and tile (64)
    boundaries; Nq > 1 rows sit at the last Nq positions of each request."""
    lens = (3, 16, 17, 63, 64, 65, 127, 129, 1000, 1023, 1024, 1025)
    shape = ai.PagedShape(12, 8, 2, Nq, 1100, 128, 16, dtype, causal, 0, None, lens, 1, 5)
    check(attn, oracle_mod, shape, 101, Nq * 2 + int(causal))


@pytest.mark.parametrize("window", [1, 50, 200, 5000])
def test_window(attn, oracle_mod, window):
    """Sliding window: the first tile starts below the window on a page
    boundary; keys below the window are masked per key."""
    shape = ai.PagedShape(6, 8, 1, 2, 4000, 64, 16, "fp16", True, window, None, None, 2, 3)
    check(attn, oracle_mod, shape, 102, window % 97)


@pytest.mark.parametrize("Hq,Hkv,Nq,max_len", [(32, 1, 1, 9000), (16, 2, 4, 6000), (4, 4, 1, 20000)])
def test_merge_paths(attn, oracle_mod, Hq, Hkv, Nq, max_len):
    """Groups of 32 rows over many chunks (the separate merge kernel) and
    small groups (the merge done by the last CTA of each group to finish)."""
    shape = ai.PagedShape(3, Hq, Hkv, Nq, max_len, 128, 16, "bf16", True, 0, None, None, max_len // 2, 2)
    check(attn, oracle_mod, shape, 103, Hq + Nq)


def test_matches_flat_cache_bitwise(attn):
    """With every request at the full length and the same chunk plan (32
    requests of 2048 tokens: one chunk each, flat and paged alike), the
    paged call computes the same tiles as the flat call on the gathered
    cache: identical bits."""
    B, L = 32, 2048
    assert attn.attn_fwd_decode_plan(B, 32, 8, 1, L, 128, False, 152, 2) == \
        attn.attn_fwd_decode_plan(B, 32, 8, 1, L, 128, True, 152, 2)
    shape = ai.PagedShape(B, 32, 8, 1, L, 128, 16, "bf16", True, 0, None, (L,) * B, 1, 0)
    q, k, v, table, lens = ai.make_paged(shape, 104, 0)
    o, lse = run_paged(attn, shape, q, k, v, table, lens)
    idx = table.long()  # (B, pages)
    kf = k[idx].permute(0, 2, 1, 3, 4).reshape(B, 8, L, 128)
    vf = v[idx].permute(0, 2, 1, 3, 4).reshape(B, 8, L, 128)
    flat = ai.AttnShape(B, 32, 8, 1, L, 128, "bf16", True)
    nb = attn.attn_fwd_workspace_bytes(B, 32, 8, 1, L, 128)
    of, lf = pu.run_cuda(flat, q, kf, vf, workspace=torch.empty(nb, dtype=torch.uint8, device="cuda:0"))
    assert torch.equal(o.cpu(), of.cpu())
    assert torch.equal(lse.cpu(), lf.cpu())


def test_poisoned_tail_is_not_used(attn, oracle_mod):
    """One request per page size whose last page is nearly empty: the NaN
    slots after the length share the tile with live keys."""
    for ps in (8, 64, 256):
        shape = ai.PagedShape(2, 4, 4, 1, 700, 64, ps, "fp16", False, 0, None, (ps + 1, 641), 1, 0)
        q, k, v, table, lens, o, lse = check(attn, oracle_mod, shape, 105, ps)
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_bad_page_index_reported(attn):
    """A table entry outside the pool: the kernel reads zeros for that page,
    finishes, and the status word reports ATTN_ERR_DEVICE_ARG once."""
    shape = ai.PagedShape(2, 8, 2, 1, 300, 64, 16, "bf16", True, 0, None, (300, 200), 1, 0)
    q, k, v, table, lens = ai.make_paged(shape, 106, 0)
    table = table.clone()
    table[1, 3] = k.shape[0] + 5
    dev = torch.device("cuda:0")
    need = attn.attn_fwd_paged_workspace_bytes(2, 8, 2, 1, 300, 64)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    attn.flash_attn_paged(q.to(dev), k.to(dev), v.to(dev), table.to(dev), lens.to(dev), 300, workspace=ws)
    assert attn.device_status() == attn.ATTN_ERR_DEVICE_ARG
    assert attn.device_status() == attn.ATTN_OK  # read and cleared
    table[1, 3] = -2
    attn.flash_attn_paged(q.to(dev), k.to(dev), v.to(dev), table.to(dev), lens.to(dev), 300, workspace=ws)
    assert attn.device_status() == attn.ATTN_ERR_DEVICE_ARG


def test_bad_length_reported(attn):
    """A length above max_seq_len, and a causal length below Nq, are clamped
    by the kernel and reported."""
    shape = ai.PagedShape(2, 8, 2, 2, 300, 64, 16, "bf16", True, 0, None, (300, 200), 1, 0)
    q, k, v, table, lens = ai.make_paged(shape, 107, 0)
    dev = torch.device("cuda:0")
    ws = torch.empty(attn.attn_fwd_paged_workspace_bytes(2, 8, 2, 2, 300, 64), dtype=torch.uint8, device=dev)
    for bad in (301, 1, 0, -4):
        l2 = lens.clone()
        l2[1] = bad
        attn.flash_attn_paged(q.to(dev), k.to(dev), v.to(dev), table.to(dev), l2.to(dev), 300, workspace=ws)
        assert attn.device_status() == attn.ATTN_ERR_DEVICE_ARG, bad


def test_host_errors(attn):
    """Workspace too small for the split-KV path (a group too large for it
    takes the prefill path instead: tests/test_paged_prefill_gpu.py)."""
    dev = torch.device("cuda:0")
    assert attn.attn_fwd_paged_path(1, 8, 1, 8, 256, 64) == attn.ATTN_PATH_PREFILL
    shape = ai.PagedShape(1, 8, 1, 2, 256, 64, 16, "fp16", True, 0, None, (256,), 1, 0)
    q, k, v, table, lens = ai.make_paged(shape, 108, 1)
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_paged(q.to(dev), k.to(dev), v.to(dev), table.to(dev), lens.to(dev), 256,
                              workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG


def test_graph_replay_with_new_lengths(attn, oracle_mod):
    """The lengths and table are read on the device: a captured graph replays
    correctly after they change in place (a decode loop's next step)."""
    shape = ai.PagedShape(4, 16, 4, 1, 2048, 128, 16, "bf16", True, 0, None, None, 100, 4)
    q, k, v, table, lens = ai.make_paged(shape, 109, 0)
    dev = torch.device("cuda:0")
    qd, kd, vd, td, ld = (t.to(dev) for t in (q, k, v, table, lens))
    ws = torch.empty(attn.attn_fwd_paged_workspace_bytes(4, 16, 4, 1, 2048, 128), dtype=torch.uint8, device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((4, 16, 1), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        attn.flash_attn_paged(qd, kd, vd, td, ld, 2048, out=o, lse=lse, workspace=ws)  # warm-up
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            attn.flash_attn_paged(qd, kd, vd, td, ld, 2048, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    for step in range(3):
        new = torch.clamp(lens - 37 * step, min=1)
        ld.copy_(new.to(dev))
        g.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle_mod.attention_paged(q, k, v, table, new, True)
        pu.compare("bf16", o.float().cpu().numpy(), o_ref, lse.cpu().numpy(), lse_ref, f"replay {step}")


@pytest.mark.parametrize("idx", [0, 1])
def test_workload_full_size(attn, oracle_mod, idx):
    """The benchmark's paged_decode calls at full size, every row against the
    oracle."""
    shape, cid, layer = ai.workload_calls("paged_decode")[idx]
    check(attn, oracle_mod, shape, cid, layer,
          config=f"C-dec paged_decode B{shape.B} Hq32 Hkv8 Nq1 L{shape.max_seq_len} ps16 d128 causal", strict=True)


def test_paged_plan(attn):
    """The paged plan keeps two CTAs per SM and caps the keys per chunk
    (lengths are known only on the device): the ragged benchmark call keeps
    the fused merge, the group too large for the split-KV kernel takes the
    prefill path, and a full-length call plans more chunks than the flat
    call (one long chunk per SM), so it needs more scratch."""
    assert attn.attn_fwd_paged_path(32, 32, 8, 1, 8192, 128) == attn.ATTN_PATH_SPLIT_KV_FUSED
    assert attn.attn_fwd_paged_path(1, 8, 1, 8, 256, 64) == attn.ATTN_PATH_PREFILL
    assert attn.attn_fwd_paged_path(4, 32, 8, 1, 8192, 128) == attn.attn_fwd_path(4, 32, 8, 1, 8192, 128, True)
    assert attn.attn_fwd_paged_workspace_bytes(4, 32, 8, 1, 8192, 128) > \
        attn.attn_fwd_workspace_bytes(4, 32, 8, 1, 8192, 128)
    assert attn.attn_fwd_paged_workspace_bytes(32, 32, 8, 1, 8192, 128) == \
        attn.attn_fwd_workspace_bytes(32, 32, 8, 1, 8192, 128)  # 4 chunks of 2048 keys either way
