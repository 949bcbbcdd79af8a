"""The split-KV plan (attn_fwd_decode_plan, no device work), on CPU.

cruxr.ai "FlashDecoding": with few query rows the keys are cut into chunks
processed in parallel, each giving a partial (max, sum, weighted V), then
merged.  The planner picks the chunk count that minimises (waves of resident
CTAs) x (K/V tiles per CTA + 2), rounds the chunk to whole 64-key tiles, and
for paged calls also caps a chunk at 32 tiles.  These tests check the plan
against those statements and against the grids the GB300 captures showed."""
import math

import pytest

KEYS = 64


@pytest.fixture(scope="module")
def attn():
    import tiled_attention_forward_fwd_gb300 as m

    m.lib()
    return m


def plan(attn, B, Hq, Hkv, Nq, Nk, d, paged=False, sms=152, per_sm=2):
    return attn.attn_fwd_decode_plan(B, Hq, Hkv, Nq, Nk, d, paged, sms, per_sm)


CASES = [(4, 32, 8, 1, 8192, 128), (4, 32, 1, 1, 8192, 128), (1, 8, 1, 3, 2000, 64), (2, 8, 2, 1, 700, 128),
         (32, 32, 8, 1, 8192, 128), (1, 32, 1, 1, 100000, 128), (8, 4, 4, 1, 65, 64), (3, 16, 2, 2, 6000, 64)]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", CASES)
@pytest.mark.parametrize("paged", [False, True])
def test_chunks_cover_keys(attn, B, Hq, Hkv, Nq, Nk, d, paged):
    p = plan(attn, B, Hq, Hkv, Nq, Nk, d, paged)
    assert p is not None
    n, ck = p["nchunks"], p["chunk_keys"]
    assert ck % KEYS == 0 and ck > 0
    assert (n - 1) * ck < Nk <= n * ck  # every key in exactly one chunk, no empty chunk at the end
    if paged:
        assert ck <= 32 * KEYS or n == 1024


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", CASES)
@pytest.mark.parametrize("sms,per_sm", [(152, 2), (152, 1), (148, 2), (10, 3)])
def test_cost_minimum(attn, B, Hq, Hkv, Nq, Nk, d, sms, per_sm):
    """The flat plan's chunk count minimises waves x (tiles per CTA + 2)
    over 1..min(tiles, 1024, 4 * slots / groups + 1) (ties: fewer chunks),
    before rounding the chunk to whole tiles."""
    p = plan(attn, B, Hq, Hkv, Nq, Nk, d, False, sms, per_sm)
    units, slots, tiles = B * Hkv, sms * per_sm, math.ceil(Nk / KEYS)
    cands = range(1, min(tiles, 1024, 4 * slots // units + 1) + 1)
    cost = {n: math.ceil(units * n / slots) * (math.ceil(tiles / n) + 2) for n in cands}
    best = min(cands, key=lambda n: (cost[n], n))
    ck = math.ceil(math.ceil(Nk / best) / KEYS) * KEYS
    assert p["chunk_keys"] == ck and p["nchunks"] == math.ceil(Nk / ck)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", CASES)
def test_merge_and_workspace(attn, B, Hq, Hkv, Nq, Nk, d):
    p = plan(attn, B, Hq, Hkv, Nq, Nk, d)
    n, R = p["nchunks"], (Hq // Hkv) * Nq
    assert p["fused"] == (1 if R * n * d <= 8192 else 0)
    part = B * Hq * Nq * n * (d + 1) * 4  # normalised partial O and its log2 LSE per (row, chunk)
    assert p["flag_off"] == (part + 15) // 16 * 16
    assert p["bytes"] == p["flag_off"] + B * Hkv * 8  # one tagged 64-bit arrival counter per group


def test_paged_cap_splits_long_requests(attn):
    flat = plan(attn, 32, 32, 8, 1, 8192, 128)
    paged = plan(attn, 32, 32, 8, 1, 8192, 128, True)
    assert flat["nchunks"] == 1 and paged["nchunks"] == 4 and paged["chunk_keys"] == 2048
    # a call that already splits finely plans the same either way
    assert plan(attn, 4, 32, 8, 1, 8192, 128) == plan(attn, 4, 32, 8, 1, 8192, 128, True)


def test_plans_seen_on_gb300(attn):
    """The mqa_decode captures on 152 SMs showed grids (9, 32) and (32, 4):
    9 chunks per group at Hkv = 8 (2 CTAs per SM), 32 at Hkv = 1 (1 CTA)."""
    assert plan(attn, 4, 32, 8, 1, 8192, 128, False, 152, 2)["nchunks"] == 9
    assert plan(attn, 4, 32, 1, 1, 8192, 128, False, 152, 1)["nchunks"] == 32


def test_shapes_without_split_path(attn):
    assert plan(attn, 1, 8, 1, 8, 4096, 128) is None       # 64 rows per group
    assert plan(attn, 65536, 8, 1, 1, 4096, 128) is None   # grid.y limit on B * Hkv
    assert plan(attn, 1, 8, 1, 1, 4096, 96) is None        # head dim
    assert plan(attn, 1, 8, 1, 1, 4096, 128, sms=0) is None
