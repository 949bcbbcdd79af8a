"""The prefill kernel's schedule, read through the C ABI without a GPU
(attn_fwd_prefill_visits), checked against first principles.

Lab 02, "La estructura del kernel" (one program per batch x head and query
tile) and the cruxr.ai "FlashAttention" loop (outer over Q blocks, inner over
K/V blocks): the output splits into independent query tiles, and each walks
the K/V tiles that hold at least one unmasked key of its rows.  Under the causal mask (bottom-right aligned when
Nq < Nk) and the sliding window, a K/V tile whose every key is masked for
every row of the tile adds nothing and is skipped.  So, whatever the item
shape, the launch must compute every (head, query tile, live K/V tile)
product exactly once and no product of a fully masked tile.  The live set
here comes from a brute-force mask over every (row, key), not from the
kernel's range arithmetic."""
import numpy as np
import pytest

BM = BN = 128
SCHED_PLAIN, SCHED_SPLIT, SCHED_HALVES = 0, 1, 2
PAIR_ROWS, PAIR_HEADS, PAIR_SINGLE, PAIR_HALVES = 0, 1, 2, 3


@pytest.fixture(scope="module")
def attn():
    import tiled_attention_forward_fwd_gb300 as m

    m.lib()
    return m


def live_tiles(Nq, Nk, causal, window):
    """bool [row tiles, K/V tiles]: the tile pair holds an unmasked (row, key)."""
    i = np.arange(Nq)[:, None] + (Nk - Nq)  # row position in key coordinates
    k = np.arange(Nk)[None, :]
    keep = np.ones((Nq, Nk), dtype=bool)
    if causal:
        keep &= k <= i
        if window > 0:
            keep &= k > i - window
    nr, nk = -(-Nq // BM), -(-Nk // BN)
    pad = np.zeros((nr * BM, nk * BN), dtype=bool)
    pad[:Nq, :Nk] = keep
    return pad.reshape(nr, BM, nk, BN).any(axis=(1, 3))


def check(attn, B, Hq, Hkv, Nq, Nk, d, causal=False, window=0, ws=False, sms=152):
    got = attn.attn_fwd_prefill_visits(B, Hq, Hkv, Nq, Nk, d, causal, window, ws, sms)
    assert got is not None, "shape should take a prefill path"
    (grid, sched, pair, n_items), v = got
    cta, item, slot, bh, row0, j = (v[:, c] for c in range(6))
    assert 0 < grid <= sms
    assert cta.min() >= 0 and cta.max() < grid
    assert item.min() >= 0 and item.max() < n_items

    # every live (head, row tile, K/V tile) exactly once, nothing else
    live = live_tiles(Nq, Nk, causal, window)
    assert (row0 % BM == 0).all()
    key = (bh.astype(np.int64) * live.shape[0] + row0 // BM) * live.shape[1] + j
    assert len(np.unique(key)) == len(key), "a product is computed twice"
    want = np.flatnonzero(np.tile(live.reshape(-1), B * Hq))
    np.testing.assert_array_equal(np.sort(key), want)

    # item shapes
    for it in np.unique(item):
        sel = item == it
        tiles = sorted(set(zip(slot[sel].tolist(), bh[sel].tolist(), row0[sel].tolist())))
        if pair == PAIR_HEADS:
            assert Hq // Hkv % 2 == 0
            for (s, h, r), (s2, h2, r2) in zip(tiles, tiles[1:]):
                assert s2 == s + 1 and r2 == r and h2 == h + 1 and h % 2 == 0
        elif pair == PAIR_ROWS:
            for (s, h, r), (s2, h2, r2) in zip(tiles, tiles[1:]):
                assert s2 == s + 1 and h2 == h and r2 == r + BM and (r // BM) % 2 == 0
        else:
            assert len({(h, r) for _, h, r in tiles}) == 1, "one query tile per item"

    if sched == SCHED_HALVES:
        assert pair == PAIR_HALVES
        for it in np.unique(item):
            sel = item == it
            js, ss = j[sel], slot[sel]
            n = len(js)
            # tile 0 takes the first ceil half of the live K/V tiles, tile 1 the rest
            assert (ss == 0).sum() == (n + 1) // 2
            assert js[ss == 0].max(initial=-1) < js[ss == 1].min(initial=1 << 30)
            # the ring alternates the halves: 0, 1, 0, 1, ..., then tile 0's last
            n1 = (ss == 1).sum()
            assert ss[:2 * n1].tolist() == [0, 1] * n1
            assert (np.diff(js[ss == 0]) == 1).all() and (np.diff(js[ss == 1]) == 1).all()
    else:
        # union order: each K/V tile loaded once per piece, ascending
        for c in np.unique(cta):
            sel = cta == c
            for it in np.unique(item[sel]):
                js = j[sel & (item == it)]
                u = np.unique(js)
                assert np.array_equal(np.sort(js, kind="stable"), js)
                assert (np.diff(u) == 1).all()

    if sched == SCHED_SPLIT:
        # stream-K: ring steps (distinct (item, K/V tile) per CTA) even over CTAs
        steps = np.array([len({(a, b) for a, b in zip(item[cta == c], j[cta == c])}) for c in range(grid)])
        assert steps.max() - steps.min() <= 1, steps
        # each CTA's range is contiguous in (item, K/V tile) order
        order = item.astype(np.int64) * (1 << 20) + j
        first = np.array([order[cta == c].min() for c in range(grid)])
        last = np.array([order[cta == c].max() for c in range(grid)])
        assert (first[1:] > last[:-1]).all()
    else:
        # whole items, each in one CTA, snake order across passes of `grid`
        for it in np.unique(item):
            assert len(np.unique(cta[item == it])) == 1
        per = {}
        for c, it in zip(cta.tolist(), item.tolist()):
            per.setdefault(c, [])
            if not per[c] or per[c][-1] != it:
                per[c].append(it)
        for c, its in per.items():
            for m, it in enumerate(its):
                assert it == m * grid + ((grid - 1 - c) if m % 2 else c)
    return grid, sched, pair, n_items


@pytest.mark.parametrize("causal", [False, True])
def test_mha_d64(attn, causal):
    # B=2, H=4, N=4096: 64 row tiles; consecutive pairs, or halves when causal
    # fits one wave of pairs
    g, sched, pair, _ = check(attn, 2, 4, 4, 4096, 4096, 64, causal)
    assert pair in (PAIR_ROWS, PAIR_HALVES)


@pytest.mark.parametrize("N", [3900, 4096])
def test_halves_causal(attn, N):
    g, sched, pair, n = check(attn, 1, 5, 5, N, N, 64, True)
    assert sched == SCHED_HALVES and n == 5 * (-(-N // BM))


@pytest.mark.parametrize("window", [129, 700])
def test_window(attn, window):
    _, _, pair, _ = check(attn, 1, 5, 5, 5000, 5000, 64, True, window)
    assert pair == (PAIR_SINGLE if window == 129 else PAIR_HALVES)


@pytest.mark.parametrize("Nq,Nk,causal", [(900, 900, True), (1000, 1000, False), (300, 2000, True),
                                          (130, 4500, False), (2 * 128 + 7, 2 * 128 + 7, True),
                                          (257, 257, True), (129, 641, True)])
def test_ragged(attn, Nq, Nk, causal):
    check(attn, 1, 3, 3, Nq, Nk, 64, causal)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (32, 8), (6, 2), (4, 4)])
def test_gqa_groups(attn, Hq, Hkv):
    _, _, pair, _ = check(attn, 2, Hq, Hkv, 1500, 1500, 128, True)
    if (Hq // Hkv) % 2 == 0:
        assert pair == PAIR_HEADS


@pytest.mark.parametrize("sms", [1, 7, 148])
def test_other_sm_counts(attn, sms):
    check(attn, 4, 41, 41, 2 * 128 + 7, 2 * 128 + 7, 64, True, sms=sms)
    check(attn, 1, 32, 8, 3000, 3000, 128, True, 300, sms=sms)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 4, 700), (1, 32, 8, 2000), (2, 3, 3, 1000), (1, 16, 16, 4096)])
def test_split_d128(attn, causal, B, Hq, Hkv, N):
    # with a workspace, d = 128 calls of few tile pairs split over the SMs
    grid, sched, _, items = check(attn, B, Hq, Hkv, N, N, 128, causal, ws=True)
    assert sched == SCHED_SPLIT
    assert items < 2 * 152


def test_split_not_taken(attn):
    # a window, d = 64, or two waves of pairs keep the whole-item schedule
    assert check(attn, 1, 4, 4, 700, 700, 128, True, 300, ws=True)[1] != SCHED_SPLIT
    assert check(attn, 1, 4, 4, 700, 700, 64, True, ws=True)[1] != SCHED_SPLIT
    assert check(attn, 8, 16, 16, 4096, 4096, 128, True, ws=True)[1] != SCHED_SPLIT


def test_other_paths_rejected(attn):
    assert attn.attn_fwd_prefill_visits(1, 4, 4, 100, 100, 64, False, 0, False, 152) is None  # short keys
    assert attn.attn_fwd_prefill_visits(4, 32, 8, 1, 8192, 128, False, 0, True, 152) is None  # split-KV
    assert attn.attn_fwd_prefill_visits(1, 4, 4, 700, 500, 64, True, 0, False, 152) is None  # causal Nq > Nk
    assert attn.attn_fwd_prefill_visits(1, 4, 4, 700, 700, 96, False, 0, False, 152) is None  # d
    assert attn.attn_fwd_prefill_visits(1, 4, 4, 700, 700, 64, False, 0, False, 0) is None  # sms


def test_truncated_buffer(attn):
    import ctypes

    L = attn.lib()
    info = (ctypes.c_int * 4)()
    buf = (ctypes.c_int * (6 * 3 + 6))()
    for x in range(len(buf)):
        buf[x] = -7
    n = L.attn_fwd_prefill_visits(1, 4, 4, 700, 700, 64, 1, 0, 0, 152, info, buf, 3)
    assert n > 3
    assert all(buf[x] != -7 for x in range(18)) and all(buf[x] == -7 for x in range(18, 24))


@pytest.mark.parametrize("B,Hkv,Nk,sms", [(4, 8, 8192, 152), (8, 12, 2048, 152), (23, 1, 2048, 152), (1, 1, 100, 152),
                                          (3, 5, 1000, 7), (2, 3, 130, 1)])
def test_bwd_cta_order(attn, B, Hkv, Nk, sms):
    """The backward's CTAs: every (K/V group, key tile) once; groups in bands
    of ceil(2 * sms / key tiles) (two waves of CTAs, the last band the rest);
    within a band the key tiles in order, so under a causal mask a CTA never
    starts before one with more query tiles to walk (lab 02, "La estructura
    del kernel": one program per head and tile)."""
    order = attn.attn_bwd_cta_order(B, Hkv, Nk, sms)
    zk, nkt = B * Hkv, -(-Nk // BN)
    assert order.shape == (zk * nkt, 2)
    assert len({(g, t) for g, t in order.tolist()}) == zk * nkt
    assert order[:, 0].min() == 0 and order[:, 0].max() == zk - 1 and order[:, 1].max() == nkt - 1
    band = min(zk, max(1, -(-2 * sms // nkt)))
    c = 0
    for first in range(0, zk, band):
        groups = list(range(first, min(zk, first + band)))
        part = order[c:c + len(groups) * nkt]
        c += len(groups) * nkt
        assert sorted(set(part[:, 0].tolist())) == groups
        assert (np.diff(part[:, 1]) >= 0).all()
        for t in range(nkt):
            assert sorted(part[part[:, 1] == t, 0].tolist()) == groups
    assert c == zk * nkt


def test_bwd_cta_order_bad_sizes(attn):
    assert attn.attn_bwd_cta_order(0, 1, 128, 152) is None
    assert attn.attn_bwd_cta_order(1, 1, 128, 0) is None
    assert attn.attn_bwd_cta_order(65536, 256, 1 << 20, 152) is None  # more than 2^31 CTAs
