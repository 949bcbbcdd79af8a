"""GPU parity of latent attention with absorbed queries (attn_fwd_mla, through
the C ABI) against the fp64 oracle.

cruxr.ai "Optimizaciones de Atencion", section "Multi-Head Latent Attention
(MLA)": the cache holds one latent vector c_t (d_c = 512) per token; with the
up-projections absorbed, every head's scores are q~ . c_t and its output is
sum_t P_t c_t, projected afterwards.  So the call is attention with one K/V
head whose keys and values are both the latent vectors: the oracle is
oracle.attention(q~, c, c) with Hkv = 1, d = 512, compared element by
element with the stated / derived bound of the other paths.  One test
also runs the whole latent-attention layer (absorb, attend, project) and
compares it with oracle.attention_mla, which rebuilds K and V explicitly."""
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


def latent_inputs(s: ai.AttnShape, cid: int, layer: int = 0):
    q, k, _ = ai.make_qkv(s, cid, layer)  # Hkv = 1: k is the latent cache
    return q, k


def run(attn, s, q, c4):
    o, lse = attn.flash_attn_mla(q.cuda(), c4[:, 0].cuda(), causal=s.causal, window=s.window, sm_scale=s.scale)
    assert attn.device_status() == attn.ATTN_OK
    return o, lse


def check(attn, oracle_mod, s, cid, layer=0, config=None):
    q, c4 = latent_inputs(s, cid, layer)
    o, lse = run(attn, s, q, c4)
    return pu.check_full(s, q, c4, c4, o, lse, oracle_mod, str(s), config)


def mla(B, n_h, Nq, Nk, dtype="bf16", causal=True, window=0, scale=1.0 / np.sqrt(128)):
    return ai.AttnShape(B, n_h, 1, Nq, Nk, 512, dtype, causal, window, float(scale), mla=True)


@pytest.mark.parametrize("Nk", [1, 2, 63, 64, 65, 200, 1000, 4097])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n_h", [16, 128])  # 16 rows: warp-MMA kernel; 128: tensor-core kernel
def test_ragged_keys(attn, oracle_mod, Nk, dtype, n_h):
    check(attn, oracle_mod, mla(2, n_h, 1, Nk, dtype), 170, Nk + n_h)


@pytest.mark.parametrize("B,Nk", [(76, 500), (40, 200)])
def test_one_chunk_direct_output(attn, oracle_mod, B, Nk):
    """Enough requests to fill the GPU with one key chunk each: the tensor-core
    kernel writes O and LSE itself (no workspace partials, no merge)."""
    s = mla(B, 128, 1, Nk)
    assert attn.attn_fwd_mla_workspace_bytes(B, 128, 1, Nk, 512) == 256  # no partials
    check(attn, oracle_mod, s, 176, B)


@pytest.mark.parametrize("B,n_h,Nq", [(1, 128, 1), (2, 8, 3), (1, 4, 1), (3, 20, 1), (1, 128, 4), (2, 1, 7)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300)])
def test_heads_and_queries(attn, oracle_mod, B, n_h, Nq, causal, window):
    """Rows n_h x Nq per request on both kernels (16-row blocks below 17 rows,
    128-row blocks from there; ragged last blocks), masks."""
    check(attn, oracle_mod, mla(B, n_h, Nq, 1500, "bf16", causal, window), 171, B * 100 + n_h + Nq)


def test_lse_without_output_lse(attn, oracle_mod):
    s = mla(2, 16, 1, 700)
    q, c4 = latent_inputs(s, 172)
    o, _ = attn.flash_attn_mla(q.cuda(), c4[:, 0].cuda(), causal=True, sm_scale=s.scale, return_lse=False)
    assert attn.device_status() == attn.ATTN_OK
    o_ref, _ = oracle_mod.attention(q, c4, c4, causal=True, sm_scale=s.scale)
    a_ref, _ = oracle_mod.attention(q, c4, c4.abs(), causal=True, sm_scale=s.scale)
    pu.compare(s.dtype, o.float().cpu().numpy(), o_ref, None, None, "no LSE", a_ref)


@pytest.mark.parametrize("idx", [0, 1])
def test_workload_sampled(attn, oracle_mod, idx):
    """The benchmark's step at full size (32 requests x 128 heads x 8192
    tokens; 8 requests x 4 queries): sampled rows against the oracle."""
    s, cid, layer = ai.workload_calls("mla_decode")[idx]
    q, c4 = latent_inputs(s, cid, layer)
    o, lse = run(attn, s, q, c4)
    pu.check_properties(s, c4, o, lse)
    pu.check_sampled(s, q, c4, c4, o, lse, oracle_mod, count=384, seed=idx, label=f"mla_decode[{idx}]",
                     config=f"C-mla mla_decode B{s.B} n_h{s.Hq} Nq{s.Nq} Nk{s.Nk} d_c512 causal")


def test_repeat_is_deterministic(attn):
    s = mla(4, 128, 1, 3000)
    q, c4 = latent_inputs(s, 173)
    o1, l1 = run(attn, s, q, c4)
    o2, l2 = run(attn, s, q, c4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_latent_layer_end_to_end(attn, oracle_mod):
    """Absorb, attend on the GPU, project: against oracle.attention_mla, which
    rebuilds every head's K and V from the latent.  W_K^up is a signed
    selection (each latent coordinate of head h copies one query coordinate,
    with a sign), so that the absorbed queries are exact in bf16 and the
    only rounding is the kernel's; W_V^up is dense.  The bound is the
    latent output's (pu.o_tolerance) carried through |W_V^up|."""
    B, n_h, Nq, Nk, d_h, d_c = 2, 8, 2, 900, 64, 512
    scale = 1.0 / np.sqrt(d_h)
    rng = np.random.default_rng(174)
    q = ai.normal_tensor(ai.seed_for(174, 0, "Q"), (B, n_h, Nq, d_h), "bf16").double().numpy()
    c = ai.normal_tensor(ai.seed_for(174, 0, "K"), (B, Nk, d_c), "bf16").double().numpy()
    wk = np.zeros((d_c, n_h, d_h))
    src = rng.integers(0, d_h, size=(d_c, n_h))
    sign = rng.choice([-1.0, 1.0], size=(d_c, n_h))
    for h in range(n_h):
        wk[np.arange(d_c), h, src[:, h]] = sign[:, h]
    wv = rng.standard_normal((d_c, n_h, d_h)) / np.sqrt(d_c)
    q_lat = np.einsum("bhid,chd->bhic", q, wk)  # exact: one +-q value per entry
    q_lat_t = torch.from_numpy(q_lat).to(torch.bfloat16)
    assert np.array_equal(q_lat_t.double().numpy(), q_lat)
    c_t = torch.from_numpy(c).to(torch.bfloat16)
    o_lat, lse = attn.flash_attn_mla(q_lat_t.cuda(), c_t.cuda(), causal=True, sm_scale=scale)
    assert attn.device_status() == attn.ATTN_OK
    o = np.einsum("bhic,chd->bhid", o_lat.double().cpu().numpy(), wv)
    o_ref, lse_ref = oracle_mod.attention_mla(q, c, wk.reshape(d_c, n_h * d_h), wv.reshape(d_c, n_h * d_h), True,
                                              0, scale)
    c4 = torch.from_numpy(c)[:, None]
    lat_ref, _ = oracle_mod.attention(torch.from_numpy(q_lat), c4, c4, causal=True, sm_scale=scale)
    a_ref, _ = oracle_mod.attention(torch.from_numpy(q_lat), c4, c4.abs(), causal=True, sm_scale=scale)
    tol_lat = pu.o_tolerance("bf16", lat_ref, a_ref)
    tol = np.einsum("bhic,chd->bhid", tol_lat, np.abs(wv)) + 1e-9
    err = np.abs(o - o_ref)
    assert (err <= tol).all(), (err.max(), tol[np.unravel_index(np.argmax(err - tol), err.shape)])
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= pu.TOL_LSE


def test_argument_errors(attn):
    s = mla(1, 4, 1, 100)
    q, c4 = latent_inputs(s, 175)
    qd, cd = q.cuda(), c4[:, 0].cuda()
    o = torch.empty_like(qd)
    ws = torch.empty(attn.attn_fwd_mla_workspace_bytes(1, 4, 1, 100, 512), dtype=torch.uint8, device="cuda")
    dt = attn.ATTN_DTYPE_BF16
    args = lambda **kw: dict(dict(Q_lat=qd.data_ptr(), C_lat=cd.data_ptr(), O_lat=o.data_ptr(), LSE=None, B=1, n_h=4,
                                  Nq=1, Nk=100, d_c=512, causal=1, window=0, sm_scale=0.1, dtype=dt,
                                  workspace=ws.data_ptr(), workspace_bytes=ws.numel(), stream=None), **kw)
    assert attn.attn_fwd_mla(**args()) == attn.ATTN_OK
    assert attn.attn_fwd_mla(**args(d_c=256)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_fwd_mla(**args(workspace_bytes=ws.numel() - 1)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_mla(**args(workspace=None)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_mla(**args(Nq=101)) == attn.ATTN_ERR_INVALID_ARG  # causal with more queries than keys
    assert attn.attn_fwd_mla(**args(sm_scale=float("nan"))) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_mla_workspace_bytes(1, 4, 1, 100, 256) == 0
    torch.cuda.synchronize()
    assert attn.device_status() == attn.ATTN_OK


# (requests, heads, tiles loaded before the stall): enough requests that each
# CTA holds one chunk of all 16 tiles (so that it stalls mid-chunk)
STALLS = [(152, 16, 0), (152, 16, 1), (40, 128, 0), (40, 128, 1), (40, 128, 3)]


@pytest.mark.parametrize("B,n_h,stall", STALLS)
def test_stalled_producer_times_out(attn, oracle_mod, B, n_h, stall):
    """The producer stops loading after `stall` latent tiles: the roles waiting
    for the next one run into the wait limit, the call comes back with
    ATTN_ERR_TIMEOUT, and the next call on the same buffers is right."""
    s = mla(B, n_h, 1, 1000)
    q, c4 = latent_inputs(s, 177)
    qd, cd = q.cuda(), c4[:, 0].cuda()
    try:
        attn.attn_set_wait_timeout_ns(200_000)
        attn.attn_set_test_stall(stall)
        attn.flash_attn_mla(qd, cd, causal=True, sm_scale=s.scale)
        assert attn.device_status() == attn.ATTN_ERR_TIMEOUT
        assert attn.device_status() == attn.ATTN_OK  # read and cleared
    finally:
        attn.attn_set_wait_timeout_ns(0)
        attn.attn_set_test_stall(-1)
    o, lse = run(attn, s, q, c4)
    pu.check_full(s, q, c4, c4, o, lse, oracle_mod, "after a stall")
