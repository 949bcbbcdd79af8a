"""Pins of the paged-cache oracle (oracle.attention_paged), on CPU.

The motivation page's "PagedAttention es un problema distinto" section: the
K/V cache lives in fixed-size pages, each request has a table of its pages
in token order, and attention reads keys through that table.  What a page
table means fixes these checks:

* writing a flat cache into pages (the allocator's direction: each token to
  a chosen page and slot) and reading it back through the table gives the
  flat cache, so the paged result equals the flat oracle (pinned on its own
  in test_oracle_pins.py) on each request's keys;
* where the pages sit in the pool does not matter: relabelling the pool's
  pages, and the table with them, leaves the result unchanged;
* slots that no request owns are never read (NaN there changes nothing);
* brute force in plain Python on tiny inputs.
"""
import math

import numpy as np
import pytest

import attn_inputs as ai
import oracle


def _scatter_into_pages(k, v, lens, page_size, rng, spare=2):
    """Write each request's first lens[b] tokens of a flat (B,Hkv,N,d) cache
    into randomly chosen pool pages; returns (k_pool, v_pool, table)."""
    B, Hkv, N, d = k.shape
    npages = [-(-int(n) // page_size) for n in lens]
    total = sum(npages) + spare
    order = rng.permutation(total)
    kp = np.full((total, Hkv, page_size, d), np.nan)
    vp = np.full((total, Hkv, page_size, d), np.nan)
    table = np.full((B, max(npages) + 1), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        for t in range(int(lens[b])):
            j, slot = divmod(t, page_size)
            if slot == 0:
                table[b, j] = order[nxt]
                nxt += 1
            kp[table[b, j], :, slot, :] = k[b, :, t, :]
            vp[table[b, j], :, slot, :] = v[b, :, t, :]
    return kp, vp, table


@pytest.mark.parametrize("page_size", [1, 3, 16])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
def test_scattered_cache_equals_flat(page_size, causal, window):
    rng = np.random.default_rng(7 + page_size)
    B, Hq, Hkv, Nq, N, d = 3, 4, 2, 2, 40, 8
    q = rng.standard_normal((B, Hq, Nq, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    lens = np.array([40, 17, 2])
    kp, vp, table = _scatter_into_pages(k, v, lens, page_size, rng)
    o, lse = oracle.attention_paged(q, kp, vp, table, lens, causal, window, 0.3)
    for b in range(B):
        n = int(lens[b])
        of, lf = oracle.attention(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], causal, window, 0.3)
        np.testing.assert_allclose(o[b], of[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], lf[0], rtol=0, atol=1e-13)


def test_page_relabelling_invariant():
    shape = ai.PagedShape(4, 6, 3, 3, 77, 16, 8, "fp16", True, 0, None, None, 1, 5)
    q, k, v, table, lens = ai.make_paged(shape, 91, 0)
    o, lse = oracle.attention_paged(q, k, v, table, lens, True)
    pi = np.random.default_rng(3).permutation(k.shape[0])
    k2 = np.empty(k.shape)
    v2 = np.empty(v.shape)
    k2[pi] = k.double().numpy()
    v2[pi] = v.double().numpy()
    t = table.numpy()
    t2 = np.where(t >= 0, pi[np.maximum(t, 0)], -1).astype(np.int32)
    o2, lse2 = oracle.attention_paged(q, k2, v2, t2, lens, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_unowned_slots_not_read():
    shape = ai.PagedShape(3, 4, 4, 1, 50, 8, 16, "bf16", False, 0, None, (50, 1, 33), 1, 4)
    q, k, v, table, lens = ai.make_paged(shape, 92, 0, poison=True)
    assert np.isnan(k.float().numpy()).any()
    o, lse = oracle.attention_paged(q, k, v, table, lens)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    q2, k2, v2, _, _ = ai.make_paged(shape, 92, 0, poison=False)
    o2, lse2 = oracle.attention_paged(q2, k2, v2, table, lens)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def _brute(q, kp, vp, table, lens, causal, window, scale):
    B, Hq, Nq, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, ps = len(kp[0]), len(kp[0][0])
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            for i in range(Nq):
                pos = lens[b] - Nq + i
                s = []
                for t in range(lens[b]):
                    if causal and t > pos:
                        continue
                    if window > 0 and pos - t >= window:
                        continue
                    page = table[b][t // ps]
                    kk = kp[page][kvh][t % ps]
                    s.append((scale * math.fsum(q[b][h][i][c] * kk[c] for c in range(d)), page, t % ps))
                m = max(x[0] for x in s)
                w = [math.exp(x[0] - m) for x in s]
                l = math.fsum(w)
                for c in range(d):
                    O[b, h, i, c] = math.fsum(wj * vp[pg][kvh][sl][c] for wj, (_, pg, sl) in zip(w, s)) / l
                L[b, h, i] = m + math.log(l)
    return O, L


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 3)])
def test_brute_force_tiny(causal, window):
    shape = ai.PagedShape(2, 4, 2, 2, 13, 4, 4, "fp16", causal, window, 0.7, (13, 6), 1, 2)
    q, k, v, table, lens = ai.make_paged(shape, 93, int(causal) + window)
    o, lse = oracle.attention_paged(q, k, v, table, lens, causal, window, 0.7)
    ob, lb = _brute(q.double().tolist(), k.double().tolist(), v.double().tolist(), table.tolist(),
                    lens.tolist(), causal, window, 0.7)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-13)


def test_bad_tables_rejected():
    q = np.zeros((1, 1, 1, 4))
    kp = np.zeros((2, 1, 4, 4))
    with pytest.raises(ValueError):
        oracle.attention_paged(q, kp, kp, [[0, 2]], [8])  # page 2 is outside the pool
    with pytest.raises(ValueError):
        oracle.attention_paged(q, kp, kp, [[0, 1]], [0])  # empty request
    with pytest.raises(ValueError):
        oracle.attention_paged(q, kp, kp, [[0, 1]], [9])  # longer than its table
    # entries past the request's pages are not read
    oracle.attention_paged(q, kp, kp, [[1, -5]], [4])


def test_generator_layout():
    """make_paged: every request's pages are distinct, table entries past its
    pages are -1, and exactly the unowned slots are NaN."""
    shape = ai.PagedShape(5, 2, 2, 1, 70, 8, 16, "fp16", True, 0, None, None, 1, 3)
    q, k, v, table, lens = ai.make_paged(shape, 94, 0)
    t = table.numpy()
    used = [int(p) for b in range(5) for p in t[b, :-(-int(lens[b]) // 16)]]
    assert len(used) == len(set(used)) == k.shape[0] - 3
    for b in range(5):
        npg = -(-int(lens[b]) // 16)
        assert (t[b, npg:] == -1).all()
        last = t[b, npg - 1]
        fill = int(lens[b]) - (npg - 1) * 16
        assert not np.isnan(k[last, :, :fill].float().numpy()).any()
        assert np.isnan(k[last, :, fill:].float().numpy()).all()
    spare = sorted(set(range(k.shape[0])) - set(used))
    assert np.isnan(v[spare].float().numpy()).all()
