"""Prefill with the stream-K split (d = 128, a workspace given, no window,
fewer tile pairs than two waves of SMs): every CTA takes an even share of K/V tile
steps, and an item cut between CTAs is merged from the partial (O, m, l) of
each piece by the CTA holding its first steps.  Parity with the fp64 oracle,
agreement with the unsplit kernel, stale workspaces, and the cases the split
leaves to the plain kernel."""
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


def _ws(attn, s, fill=None):
    n = attn.attn_fwd_workspace_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d)
    assert n > 0, s
    if fill is None:
        return torch.empty(n, dtype=torch.uint8, device="cuda")
    return torch.full((n,), fill, dtype=torch.uint8, device="cuda")


def _split_path(attn, s):
    return attn.attn_fwd_path(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, True)


@pytest.mark.parametrize("N", [256, 1024, 4096])
@pytest.mark.parametrize("causal", [False, True])
def test_b2h4_split(attn, oracle_mod, N, causal):
    """The MHA B=2, H=4 sizes at d = 128."""
    shape = ai.AttnShape(2, 4, 4, N, N, 128, "bf16", causal)
    assert _split_path(attn, shape) == attn.ATTN_PATH_PREFILL_SPLIT
    q, k, v = ai.make_qkv(shape, config_id=73, layer=N)
    o, lse = pu.run_cuda(shape, q, k, v, workspace=_ws(attn, shape))
    if shape.Nq <= 1024:
        pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"split {shape}")
    else:
        pu.check_sampled(shape, q, k, v, o, lse, oracle_mod, count=384, label=f"split {shape}")
        # the unsplit kernel on the same inputs: same math, another summation order
        o2, lse2 = pu.run_cuda(shape, q, k, v)
        assert (o.float() - o2.float()).abs().max().item() <= 1.6e-2
        assert (lse - lse2).abs().max().item() <= 1e-4


SHAPES = [  # B, Hq, Hkv, Nq, Nk, d, dtype, causal
    (1, 2, 2, 129, 129, 128, "fp16", False),
    (1, 2, 2, 129, 129, 128, "fp16", True),
    (1, 4, 4, 700, 700, 128, "fp16", True),
    (2, 3, 3, 513, 513, 128, "bf16", False),
    (2, 3, 3, 513, 513, 128, "bf16", True),
    (1, 8, 1, 300, 777, 128, "bf16", True),
    (2, 4, 2, 1000, 1000, 128, "bf16", True),
    (1, 6, 2, 384, 384, 128, "fp16", True),
    (1, 2, 2, 2048, 2048, 128, "fp16", False),
    (1, 2, 1, 1500, 1500, 128, "bf16", True),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dtype,causal", SHAPES)
def test_split_shapes(attn, oracle_mod, B, Hq, Hkv, Nq, Nk, d, dtype, causal):
    """Ragged row and key counts, GQA groups that pair heads (even) and rows
    (odd), Nq < Nk (bottom-right causal)."""
    shape = ai.AttnShape(B, Hq, Hkv, Nq, Nk, d, dtype, causal)
    assert _split_path(attn, shape) == attn.ATTN_PATH_PREFILL_SPLIT
    q, k, v = ai.make_qkv(shape, config_id=70, layer=Nq)
    o, lse = pu.run_cuda(shape, q, k, v, workspace=_ws(attn, shape))
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"split {shape}")


def test_stale_workspace_and_reuse(attn, oracle_mod):
    """A workspace full of garbage (flags included) and reused call after call
    gives the same, correct result: each launch waits for its own token."""
    shape = ai.AttnShape(2, 4, 4, 1024, 1024, 128, "fp16", True)
    q, k, v = ai.make_qkv(shape, config_id=71)
    ws = _ws(attn, shape, fill=0x7F)
    o1, l1 = pu.run_cuda(shape, q, k, v, workspace=ws)
    o2, l2 = pu.run_cuda(shape, q, k, v, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    pu.check_full(shape, q, k, v, o1, l1, oracle_mod, "stale workspace")


def test_window_takes_the_plain_kernel(attn, oracle_mod):
    """With a window the split is not used, workspace or not."""
    shape = ai.AttnShape(1, 4, 4, 700, 700, 128, "fp16", True, 200)
    q, k, v = ai.make_qkv(shape, config_id=72)
    o, lse = pu.run_cuda(shape, q, k, v, workspace=_ws(attn, shape))
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, "window with workspace")


@pytest.mark.parametrize("kind,x", [("step", 1.5), ("spike", 7.5)])
def test_split_rescale(attn, oracle_mod, kind, x):
    """Scores that grow tile by tile, so that pieces of one row see very
    different maxima and the merge rescales partials by large factors."""
    N, d = 2048, 128
    shape = ai.AttnShape(1, 2, 2, N, N, d, "fp16", False)
    ln2 = float(np.log(2.0))
    blk = torch.arange(N, dtype=torch.float64) // 128
    c = blk * x * ln2
    if kind == "spike":
        c = torch.where(torch.arange(N) % 128 == 5, c, torch.full_like(c, -30.0))
    q = torch.zeros(1, 2, N, d, dtype=torch.float64)
    q[..., 0] = d ** 0.5 * (1.0 + (torch.arange(N) % 7) / 7.0)
    k = torch.zeros(1, 2, N, d, dtype=torch.float64)
    k[..., 0] = c
    k[..., 1:] = ai.normal_tensor(86, (1, 2, N, d - 1), "f64") * 0.01
    v = ai.normal_tensor(87, (1, 2, N, d), "f64")
    q, k, v = q.half(), k.half(), v.half()
    assert _split_path(attn, shape) == attn.ATTN_PATH_PREFILL_SPLIT
    o, lse = pu.run_cuda(shape, q, k, v, workspace=_ws(attn, shape))
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"split rescale {kind} {x}")


def test_no_split_at_d64(attn):
    """At d = 64 the plain kernel is faster at every size: no workspace."""
    assert attn.attn_fwd_workspace_bytes(2, 4, 4, 4096, 4096, 64) == 0
    assert attn.attn_fwd_path(2, 4, 4, 4096, 4096, 64, True) == attn.ATTN_PATH_PREFILL
