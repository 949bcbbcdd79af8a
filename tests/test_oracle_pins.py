"""Pins for the fp64 CPU oracle: each check ties it to something other than
itself (a worked example from the pages, a closed form, an invariant, a
textbook library routine or brute force on tiny inputs)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from attn_inputs import AttnShape, make_qkv, normal_tensor
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EXACT = 1e-12


def rnd(shape, seed, scale=1.0):
    return normal_tensor(seed, shape, "f64", scale=scale).numpy()


def test_cruxr_worked_example(oracle_mod):
    """cruxr.ai worked example: s=8, d_k=4, blocks of 2, sin inputs; the tiled
    online softmax and the standard full-matrix attention agree below 1e-10."""
    g = json.load(open(os.path.join(GOLDEN, "cruxr_tiled_demo.json")))
    s, dk, blk = g["s"], g["d_k"], g["block"]
    Q = np.array(pins.sin_matrix(s, dk, g["seeds"]["Q"]))[None, None]
    K = np.array(pins.sin_matrix(s, dk, g["seeds"]["K"]))[None, None]
    V = np.array(pins.sin_matrix(s, dk, g["seeds"]["V"]))[None, None]
    O, L = oracle_mod.attention(Q, K, V, causal=False, sm_scale=1.0 / math.sqrt(dk))
    Ot, Lt = pins.tiled_online_attention(Q, K, V, block_q=blk, block_k=blk)
    assert np.abs(O - Ot).max() < g["claim_max_abs_difference_below"]
    assert np.abs(L - Lt).max() < g["claim_max_abs_difference_below"]
    Ob, Lb = pins.brute_attention(Q, K, V)
    assert np.abs(O - Ob).max() < 1e-14
    assert np.abs(L - Lb).max() < 1e-13


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5), (True, 1)])
@pytest.mark.parametrize("bq,bk", [(1, 1), (3, 5), (16, 7), (64, 64)])
def test_online_equals_batch(oracle_mod, causal, window, bq, bk):
    """Online softmax over any block size (1, non-divisors, whole) equals the
    batch softmax of the oracle (the recurrence is exact, not approximate)."""
    B, H, N, d = 1, 2, 37, 8
    Q, K, V = rnd((B, H, N, d), 11), rnd((B, H, N, d), 12, 2.0), rnd((B, H, N, d), 13)
    O, L = oracle_mod.attention(Q, K, V, causal=causal, window=window)
    Ot, Lt = pins.tiled_online_attention(Q, K, V, bq, bk, causal=causal, window=window)
    assert np.abs(O - Ot).max() < EXACT
    assert np.abs(L - Lt).max() < EXACT


@pytest.mark.parametrize("causal,window,Nq", [(False, 0, 9), (True, 0, 9), (True, 3, 9), (True, 0, 4),
                                              (False, 0, 1), (True, 2, 1)])
def test_brute_force_tiny(oracle_mod, causal, window, Nq):
    """Pure-Python fsum double loops on N <= 16, GQA g=2, Nq <= Nk."""
    B, Hq, Hkv, Nk, d = 2, 4, 2, 9, 5
    Q, K, V = rnd((B, Hq, Nq, d), 21), rnd((B, Hkv, Nk, d), 22), rnd((B, Hkv, Nk, d), 23)
    O, L = oracle_mod.attention(Q, K, V, causal=causal, window=window, sm_scale=0.7)
    Ob, Lb = pins.brute_attention(Q, K, V, causal=causal, window=window, sm_scale=0.7)
    assert np.abs(O - Ob).max() < 1e-13
    assert np.abs(L - Lb).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_torch_library_softmax(oracle_mod, causal):
    """Textbook routine: torch float64 softmax(Q K^T * scale + mask) @ V."""
    B, H, N, d = 1, 3, 200, 16
    Q, K, V = rnd((B, H, N, d), 31), rnd((B, H, N, d), 32), rnd((B, H, N, d), 33)
    O, L = oracle_mod.attention(Q, K, V, causal=causal)
    q, k, v = map(torch.from_numpy, (Q, K, V))
    S = q @ k.transpose(-1, -2) / math.sqrt(d)
    if causal:
        S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    P = torch.softmax(S, dim=-1)
    assert np.abs(O - (P @ v).numpy()).max() < EXACT
    assert np.abs(L - torch.logsumexp(S, dim=-1).numpy()).max() < EXACT


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 6)])
def test_identical_keys_give_mean_of_v(oracle_mod, causal, window):
    """All keys equal: every live score is the same, so O is the mean of V over
    the live set and LSE = s + ln|J|."""
    B, H, N, d = 1, 2, 23, 8
    Q, V = rnd((B, H, N, d), 41), rnd((B, H, N, d), 42)
    krow = rnd((d,), 43)
    K = np.broadcast_to(krow, (B, H, N, d)).copy()
    scale = 1.0 / math.sqrt(d)
    O, L = oracle_mod.attention(Q, K, V, causal=causal, window=window)
    for h in range(H):
        for i in range(N):
            lo = max(0, i - window + 1) if window > 0 else 0
            hi = i + 1 if causal else N
            assert np.abs(O[0, h, i] - V[0, h, lo:hi].mean(axis=0)).max() < EXACT
            s = scale * float(Q[0, h, i] @ krow)
            assert abs(L[0, h, i] - (s + math.log(hi - lo))) < EXACT


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 4)])
def test_one_hot_v_exposes_weights(oracle_mod, causal, window):
    """V = identity (d = N): O row i is the softmax weight row P[i,:].  The
    weights are >= 0, sum to 1, vanish exactly on masked keys, their ratios are
    exp(s_j - s_j') from plain dot products, and ln P[i,j] = s_j - LSE[i]."""
    N = d = 12
    Q, K = rnd((1, 1, N, d), 51), rnd((1, 1, N, d), 52)
    V = np.eye(N)[None, None]
    scale = 0.5
    O, L = oracle_mod.attention(Q, K, V, causal=causal, window=window, sm_scale=scale)
    P = O[0, 0]
    for i in range(N):
        live = [j for j in range(N) if pins.live(i, j, causal, window)]
        dead = [j for j in range(N) if j not in live]
        assert abs(P[i].sum() - 1.0) < EXACT
        assert (P[i] >= 0).all()
        assert all(P[i, j] == 0.0 for j in dead)
        s = {j: scale * float(Q[0, 0, i] @ K[0, 0, j]) for j in live}
        j0 = live[0]
        for j in live:
            assert abs(P[i, j] / P[i, j0] - math.exp(s[j] - s[j0])) < 1e-11 * max(1.0, math.exp(s[j] - s[j0]))
            assert abs(math.log(P[i, j]) - (s[j] - L[0, 0, i])) < 1e-11


def test_causal_row0_and_window1(oracle_mod):
    """Causal row 0 attends only to key 0 (O = V[0], LSE = scale q0.k0); with
    window = 1 every row attends only to itself (O = V[i], LSE = scale qi.ki)."""
    B, H, N, d = 2, 2, 17, 8
    Q, K, V = rnd((B, H, N, d), 61), rnd((B, H, N, d), 62), rnd((B, H, N, d), 63)
    scale = 1.0 / math.sqrt(d)
    O, L = oracle_mod.attention(Q, K, V, causal=True)
    assert np.abs(O[:, :, 0] - V[:, :, 0]).max() == 0.0
    assert np.abs(L[:, :, 0] - scale * np.einsum("bhc,bhc->bh", Q[:, :, 0], K[:, :, 0])).max() < EXACT
    O1, L1 = oracle_mod.attention(Q, K, V, causal=True, window=1)
    assert np.abs(O1 - V).max() == 0.0
    assert np.abs(L1 - scale * np.einsum("bhnc,bhnc->bhn", Q, K)).max() < EXACT


def test_n1_noncausal(oracle_mod):
    Q, K, V = rnd((1, 3, 1, 8), 71), rnd((1, 3, 1, 8), 72), rnd((1, 3, 1, 8), 73)
    O, L = oracle_mod.attention(Q, K, V, sm_scale=0.3)
    assert np.abs(O - V).max() == 0.0
    assert np.abs(L - 0.3 * np.einsum("bhnc,bhnc->bhn", Q, K)).max() < EXACT


def test_window_at_least_n_is_causal(oracle_mod):
    Q, K, V = rnd((1, 2, 29, 8), 81), rnd((1, 2, 29, 8), 82), rnd((1, 2, 29, 8), 83)
    Oc, Lc = oracle_mod.attention(Q, K, V, causal=True)
    for w in (29, 30, 1000):
        Ow, Lw = oracle_mod.attention(Q, K, V, causal=True, window=w)
        assert np.array_equal(Oc, Ow) and np.array_equal(Lc, Lw)
    Ow, _ = oracle_mod.attention(Q, K, V, causal=True, window=28)
    assert not np.array_equal(Oc, Ow)


@pytest.mark.parametrize("Hkv", [1, 2, 4, 8])
def test_gqa_equals_mha_on_repeated_kv(oracle_mod, Hkv):
    """GQA with Hkv heads equals MHA with each K/V head repeated g = Hq/Hkv
    times consecutively (Hkv = Hq is MHA itself, Hkv = 1 is MQA)."""
    B, Hq, N, d = 2, 8, 19, 8
    Q, K, V = rnd((B, Hq, N, d), 91), rnd((B, Hkv, N, d), 92), rnd((B, Hkv, N, d), 93)
    g = Hq // Hkv
    for causal in (False, True):
        O, L = oracle_mod.attention(Q, K, V, causal=causal)
        Om, Lm = oracle_mod.attention(Q, np.repeat(K, g, axis=1), np.repeat(V, g, axis=1), causal=causal)
        assert np.array_equal(O, Om) and np.array_equal(L, Lm)
        # and head h really reads kv head h // g (not h % Hkv): compare per head
        for h in range(Hq):
            Oh, _ = oracle_mod.attention(Q[:, h:h + 1], K[:, h // g:h // g + 1], V[:, h // g:h // g + 1],
                                         causal=causal)
            assert np.array_equal(O[:, h:h + 1], Oh)


def test_linearity_in_v_and_key_permutation(oracle_mod):
    B, H, N, d = 1, 2, 31, 8
    Q, K = rnd((B, H, N, d), 101), rnd((B, H, N, d), 102)
    V1, V2 = rnd((B, H, N, d), 103), rnd((B, H, N, d), 104)
    O1, _ = oracle_mod.attention(Q, K, V1)
    O2, _ = oracle_mod.attention(Q, K, V2)
    O12, _ = oracle_mod.attention(Q, K, V1 + V2)
    assert np.abs(O12 - (O1 + O2)).max() < EXACT
    perm = np.random.default_rng(0).permutation(N)
    Op, Lp = oracle_mod.attention(Q, K[:, :, perm], V1[:, :, perm])
    O, L = oracle_mod.attention(Q, K, V1)
    assert np.abs(Op - O).max() < EXACT and np.abs(Lp - L).max() < EXACT


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 7)])
def test_lse_bounds(oracle_mod, causal, window):
    """max_j s_j <= LSE <= max_j s_j + ln|J(i)| for every row."""
    B, H, N, d = 1, 2, 40, 16
    Q, K, V = rnd((B, H, N, d), 111), rnd((B, H, N, d), 112, 3.0), rnd((B, H, N, d), 113)
    scale = 1.0 / math.sqrt(d)
    _, L = oracle_mod.attention(Q, K, V, causal=causal, window=window)
    S = scale * np.einsum("bhic,bhjc->bhij", Q, K)
    for i in range(N):
        live = [j for j in range(N) if pins.live(i, j, causal, window)]
        smax = S[:, :, i, live].max(axis=-1)
        assert (L[:, :, i] >= smax - EXACT).all()
        assert (L[:, :, i] <= smax + math.log(len(live)) + EXACT).all()


def test_bottom_right_alignment(oracle_mod):
    """With Nq < Nk, causal query i sits at position Nk - Nq + i: its result is
    row Nk - Nq + i of the square causal problem; decode (Nq = 1) sees the
    whole cache, i.e. equals non-causal."""
    B, H, Nk, d = 1, 2, 33, 8
    Qf, K, V = rnd((B, H, Nk, d), 121), rnd((B, H, Nk, d), 122), rnd((B, H, Nk, d), 123)
    Of, Lf = oracle_mod.attention(Qf, K, V, causal=True)
    for Nq in (1, 5, 33):
        Oq, Lq = oracle_mod.attention(Qf[:, :, Nk - Nq:], K, V, causal=True)
        assert np.array_equal(Oq, Of[:, :, Nk - Nq:]) and np.array_equal(Lq, Lf[:, :, Nk - Nq:])
    O1, L1 = oracle_mod.attention(Qf[:, :, -1:], K, V, causal=True)
    On, Ln = oracle_mod.attention(Qf[:, :, -1:], K, V, causal=False)
    assert np.array_equal(O1, On) and np.array_equal(L1, Ln)


def test_empty_live_set_is_nan(oracle_mod):
    """Causal with Nq > Nk leaves the first rows with no live key: no defined
    softmax, reported as NaN / -inf so any comparison fails."""
    Q, K, V = rnd((1, 1, 6, 4), 131), rnd((1, 1, 4, 4), 132), rnd((1, 1, 4, 4), 133)
    O, L = oracle_mod.attention(Q, K, V, causal=True)
    assert np.isnan(O[0, 0, :2]).all() and np.isneginf(L[0, 0, :2]).all()
    assert np.isfinite(O[0, 0, 2:]).all()


def test_rows_entry_matches_full(oracle_mod):
    shape = AttnShape(B=2, Hq=4, Hkv=2, Nq=50, Nk=50, d=16, dtype="bf16", causal=True, window=9)
    q, k, v = make_qkv(shape, config_id=7)
    O, L = oracle_mod.attention(q, k, v, causal=True, window=9)
    ids = np.array([0, 3, 49, 50, 177, 399], dtype=np.int64)
    qr = q.reshape(-1, 16)[torch.from_numpy(ids)]
    Or, Lr = oracle_mod.attention_rows(qr, ids, k, v, B=2, Hq=4, Nq=50, causal=True, window=9)
    assert np.array_equal(Or, O.reshape(-1, 16)[ids]) and np.array_equal(Lr, L.reshape(-1)[ids])


def test_bad_args_rejected(oracle_mod):
    Q, K, V = rnd((1, 3, 4, 4), 1), rnd((1, 2, 4, 4), 2), rnd((1, 2, 4, 4), 3)
    with pytest.raises(ValueError):
        oracle_mod.attention(Q, K, V)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle_mod.attention(Q[:, :2], K, V, sm_scale=-1.0)
