"""The split-KV plan (attn_fwd_decode_plan, no device work), on CPU.

cruxr.ai "FlashDecoding": with few query rows the keys are cut into chunks
processed in parallel, each giving a partial (max, sum, weighted V), then
merged.  The planner picks the chunk count that minimises, for flat calls,
(CTAs per SM) x (K/V tiles per CTA + 6), and for paged calls (waves of
resident CTAs) x (tiles per CTA + 2) with a chunk capped at 32 tiles (int8
calls: the same without the cap); it rounds the chunk to whole 64-key
tiles.  These tests check the plan against
those statements and against the grids measured on GB300."""
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
    """The flat plan's chunk count minimises (CTAs per SM) x (tiles per CTA
    + 6) over 1..min(tiles, 1024, 4 * slots / groups + 1) (ties: fewer
    chunks), before rounding the chunk to whole tiles; the paged plan's,
    waves of resident CTAs x (tiles per CTA + 2), before its 32-tile cap."""
    units, slots, tiles = B * Hkv, sms * per_sm, math.ceil(Nk / KEYS)
    cands = range(1, min(tiles, 1024, 4 * slots // units + 1) + 1)
    for paged in (0, 1, 2):  # flat, paged, int8
        p = plan(attn, B, Hq, Hkv, Nq, Nk, d, paged, sms, per_sm)
        if paged:
            cost = {n: math.ceil(units * n / slots) * (math.ceil(tiles / n) + 2) for n in cands}
        else:
            cost = {n: math.ceil(units * n / sms) * (math.ceil(tiles / n) + 6) for n in cands}
        best = min(cands, key=lambda n: (cost[n], n))
        if paged == 1:
            best = max(best, min(math.ceil(tiles / 32), 1024))
        ck = math.ceil(math.ceil(Nk / best) / KEYS) * KEYS
        assert p["chunk_keys"] == ck and p["nchunks"] == math.ceil(Nk / ck), (paged, p, best)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d", CASES)
def test_merge_and_workspace(attn, B, Hq, Hkv, Nq, Nk, d):
    p = plan(attn, B, Hq, Hkv, Nq, Nk, d)
    n, R = p["nchunks"], (Hq // Hkv) * Nq
    assert p["fused"] == (1 if R * n * d <= 8192 else 0)
    part = B * Hq * Nq * n * (d + 1) * 4  # normalised partial O and its log2 LSE per (row, chunk)
    assert p["flag_off"] == (part + 15) // 16 * 16
    assert p["bytes"] == p["flag_off"] + B * Hkv * 8  # one tagged 64-bit arrival counter per group


def test_paged_cap_splits_long_requests(attn):
    flat = plan(attn, 152, 32, 8, 1, 8192, 128)  # 1216 groups: one chunk each fills every SM 8 times
    paged = plan(attn, 152, 32, 8, 1, 8192, 128, True)
    assert flat["nchunks"] == 1 and paged["nchunks"] == 4 and paged["chunk_keys"] == 2048


def test_plans_measured_on_gb300(attn):
    """mqa_decode on 152 SMs: 4 chunks per group at Hkv = 8 (grid (4, 32), one
    CTA per SM; measured 33.0 us against 35.1 us for the 9 chunks at two per
    SM that a wave-count model picks), 32 at Hkv = 1 (grid (32, 4)); the
    paged call of the same size keeps 9 chunks at two CTAs per SM (its
    producer issues a copy per page: 34.8 us against 47.1 us with 4)."""
    assert plan(attn, 4, 32, 8, 1, 8192, 128, False, 152, 2)["nchunks"] == 4
    assert plan(attn, 4, 32, 8, 1, 8192, 128, True, 152, 2)["nchunks"] == 9
    assert plan(attn, 4, 32, 1, 1, 8192, 128, False, 152, 1)["nchunks"] == 32
    assert plan(attn, 4, 32, 8, 1, 8192, 128, 2, 152, 2)["nchunks"] == 9  # int8: two CTAs per SM
    assert plan(attn, 4, 32, 8, 1, 8192, 128, 3, 152, 2) is None


def test_shapes_without_split_path(attn):
    assert plan(attn, 1, 8, 1, 8, 4096, 128) is None       # 64 rows per group
    assert plan(attn, 65536, 8, 1, 1, 4096, 128) is None   # grid.y limit on B * Hkv
    assert plan(attn, 1, 8, 1, 1, 4096, 96) is None        # head dim
    assert plan(attn, 1, 8, 1, 1, 4096, 128, sms=0) is None
