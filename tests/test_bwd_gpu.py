"""GPU parity of the backward pass (attn_bwd, through the C ABI) against the
fp64 oracle's gradients of the forward definition (oracle.attention_bwd,
pinned on CPU by finite differences and autograd).

The pages store the log-sum-exp "for the backward pass" (cruxr.ai
"FlashAttention: Nunca materializar la matriz de atencion"; lab 02 kernel
skeleton) and defer the backward itself; its arithmetic here is the plain
one: P recomputed from Q, K and LSE; dV = P^T dO; dS = P o (dO V^T - D) with
D = rowsum(dO o O); dK = scale dS^T Q; dQ = scale dS K; P and dS rounded to
the input dtype before their products, as the forward rounds P.

The forward (the library's own kernel) gives O and LSE for each case.  The
bound per element is what an exact kernel following that arithmetic can be
off by (derived below, in fp64): the 16-bit P and dS, D taken from the
16-bit O, fp32 accumulation, and the 16-bit output."""
import numpy as np
import pytest
import torch

import attn_inputs as ai

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

U = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}  # unit roundoff of the 16-bit P and dS


@pytest.fixture(scope="module")
def attn():
    import tiled_attention_forward_fwd_gb300 as m

    m.lib()
    return m


def half_ulp(dtype, x):
    bits = 11 if dtype == "fp16" else 8
    tiny = 2.0 ** -14 if dtype == "fp16" else 2.0 ** -126
    ax = np.maximum(np.abs(x), tiny)
    return 0.5 * 2.0 ** (np.floor(np.log2(ax)) - (bits - 1))


def bwd_bounds(s, q, k, v, do, o16):
    """Elementwise bounds on |dX_gpu - dX_oracle| for X = Q, K, V."""
    u = U[s.dtype]
    Q, K, V, G, O16 = (t.double().numpy() for t in (q, k, v, do, o16))
    g = s.Hq // s.Hkv
    bq = np.zeros_like(Q)
    bk = np.zeros_like(K)
    bv = np.zeros_like(V)
    pos = (s.Nk - s.Nq) + np.arange(s.Nq)[:, None]
    j = np.arange(s.Nk)[None, :]
    live = np.ones((s.Nq, s.Nk), bool)
    if s.causal:
        live &= j <= pos
        if s.window > 0:
            live &= pos - j < s.window
    for b in range(s.B):
        for h in range(s.Hq):
            kv = h // g
            S = s.scale * Q[b, h] @ K[b, kv].T
            S = np.where(live, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            E = np.where(live, np.exp(S - m), 0.0)
            P = E / np.maximum(E.sum(axis=1, keepdims=True), 1e-300)
            dP = G[b, h] @ V[b, kv].T
            D = (P * dP).sum(axis=1, keepdims=True)
            D16 = (G[b, h] * O16[b, h]).sum(axis=1, keepdims=True)
            dS = P * (dP - D16)
            dPabs = np.abs(G[b, h]) @ np.abs(V[b, kv]).T
            dd = np.abs(G[b, h] * O16[b, h]).sum(axis=1, keepdims=True)
            # error of the kernel's dS: its own rounding, P's rounding (and
            # the fp32 LSE), D from the rounded O, fp32 sums in dP and D
            e_ds = u * np.abs(dS) + (u + 1e-5) * P * np.abs(dP - D16) + P * np.abs(D16 - D) \
                + P * 1e-5 * (dPabs + dd)
            bv[b, kv] += (u + 1e-5) * P.T @ np.abs(G[b, h])
            bk[b, kv] += s.scale * e_ds.T @ np.abs(Q[b, h])
            bq[b, h] += s.scale * e_ds @ np.abs(K[b, kv])
    return bq, bk, bv


def check(attn, oracle_mod, s, cid, layer=0):
    q, k, v = ai.make_qkv(s, config_id=cid, layer=layer)
    do = ai.normal_tensor(ai.seed_for(cid, layer, "G"), tuple(q.shape), s.dtype)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.flash_attn_forward(qd, kd, vd, causal=s.causal, window=s.window, sm_scale=s.scale)
    dq, dk, dv = attn.flash_attn_backward(qd, kd, vd, o, lse, dod, s.causal, s.window, s.scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.ATTN_OK
    rq, rk, rv = oracle_mod.attention_bwd(q, k, v, do, causal=s.causal, window=s.window, sm_scale=s.scale)
    bq, bk, bv = bwd_bounds(s, q, k, v, do, o.cpu())
    stats = {}
    for name, got, ref, bnd in (("dQ", dq, rq, bq), ("dK", dk, rk, bk), ("dV", dv, rv, bv)):
        got = got.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all(), name
        err = np.abs(got - ref)
        tol = bnd + half_ulp(s.dtype, np.abs(ref) + bnd) + 1e-5 * (np.abs(ref) + bnd) + 1e-6
        worst = np.unravel_index(np.argmax(err - tol), err.shape)
        assert (err <= tol).all(), f"{s} {name}: error {err[worst]:.3e} > bound {tol[worst]:.3e} at {worst}, " \
                                   f"|ref| {abs(ref[worst]):.3e}"
        # the bound is not vacuous: a few per cent of the gradient's scale at most
        assert tol.max() <= 0.05 * np.abs(ref).max() + 1e-3, (name, tol.max(), np.abs(ref).max())
        stats[name] = (float(err.max()), float(np.abs(ref).max()))
    return stats


CASES = [
    ai.AttnShape(1, 2, 2, 256, 256, 64, "fp16", False),
    ai.AttnShape(1, 2, 2, 256, 256, 64, "fp16", True),
    ai.AttnShape(2, 4, 2, 300, 300, 128, "bf16", True),      # GQA, ragged
    ai.AttnShape(1, 2, 1, 1, 1, 64, "bf16", False),          # one row, one key
    ai.AttnShape(1, 4, 4, 200, 500, 128, "bf16", True),      # Nq < Nk (bottom-right)
    ai.AttnShape(1, 2, 2, 700, 700, 64, "fp16", True, 128),  # window
    ai.AttnShape(1, 2, 2, 700, 700, 128, "bf16", True, 300),
    ai.AttnShape(1, 8, 1, 384, 384, 128, "bf16", False),     # MQA
    ai.AttnShape(2, 2, 2, 129, 129, 128, "fp16", True),      # one key past a tile
    # 23 K/V groups x 16 key tiles: on a 152-SM part the CTAs form bands of
    # ceil(304 / 16) = 19 groups, the last band holding 4
    ai.AttnShape(23, 1, 1, 2048, 2048, 64, "bf16", True),
]


@pytest.mark.parametrize("s", CASES, ids=[f"B{c.B}H{c.Hq}/{c.Hkv}N{c.Nq}x{c.Nk}d{c.d}{c.dtype}c{int(c.causal)}"
                                          f"w{c.window}" for c in CASES])
def test_gradients(attn, oracle_mod, s):
    check(attn, oracle_mod, s, 160, s.Nq % 97)


def test_errors(attn):
    dev = "cuda"
    q = torch.zeros(1, 2, 64, 64, device=dev, dtype=torch.float16)
    lse = torch.zeros(1, 2, 64, device=dev)
    with pytest.raises(attn.AttnError) as e:
        attn.flash_attn_backward(q, q, q, q, lse, q, workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.status == attn.ATTN_ERR_INVALID_ARG
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("d", [64, 128])
def test_wait_limit_then_recovery(attn, oracle_mod, d):
    """Every wait of the backward is bounded: with a 1 ns limit (a wait that
    polls more than once gives up) the call comes back with ATTN_OK or
    ATTN_ERR_TIMEOUT, and with the default limit the next call on the same
    buffers matches the oracle."""
    s = ai.AttnShape(1, 4, 2, 300, 300, d, "bf16", True)
    q, k, v = ai.make_qkv(s, config_id=190)
    do = ai.normal_tensor(ai.seed_for(190, 0, "G"), tuple(q.shape), s.dtype)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = attn.flash_attn_forward(qd, kd, vd, causal=True)
    try:
        attn.attn_set_wait_timeout_ns(1)
        for _ in range(3):
            attn.flash_attn_backward(qd, kd, vd, o, lse, dod, causal=True)
            st = attn.device_status()
            assert st in (attn.ATTN_OK, attn.ATTN_ERR_TIMEOUT), attn.attn_status_string(st)
    finally:
        attn.attn_set_wait_timeout_ns(0)
    check(attn, oracle_mod, s, 190)
