"""GPU parity of the prefill kernel's item shapes, through the C ABI, against
the fp64 oracle.  The host picks, per call: two heads of a GQA group (even
group sizes); one tile per item when the tiles are few, with its K/V tiles
split between the two softmax warpgroups ("halves": interleaved ring, merge
of the two partial results in the CTA) when the longest tile has at least 4
K/V tiles, else whole; consecutive row tiles otherwise.  Each case below is
sized to land on one of them on a 152-SM GB300 (the item shape changes only
the schedule, never the result)."""
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


def _check(shape, oracle_mod, cid, layer=0):
    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    o, lse = pu.run_cuda(shape, q, k, v)
    pu.check_full(shape, q, k, v, o, lse, oracle_mod, f"{shape}")


@pytest.mark.parametrize("N", [3900, 4096])
def test_halves_causal_one_wave(attn, oracle_mod, N):
    """5 heads x 31 or 32 row tiles, causal: too many tiles for one per SM,
    but pairs would fit one wave; halves items, two waves, tile lengths 1-32
    (length 1: the second warpgroup has no half; odd lengths: unequal
    halves)."""
    _check(ai.AttnShape(1, 5, 5, N, N, 64, "fp16", True), oracle_mod, 80, N)


@pytest.mark.parametrize("window", [129, 700])
def test_window_few_tiles(attn, oracle_mod, window):
    """A window of 129 leaves every tile at most 3 K/V tiles: whole single
    tiles; 700 gives up to 7: halves."""
    _check(ai.AttnShape(1, 5, 5, 5000, 5000, 64, "bf16", True, window), oracle_mod, 81, window)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(3, 3), (6, 2)])
def test_halves_odd_groups_d128(attn, oracle_mod, causal, Hq, Hkv):
    """Few tiles (every tile gets its own SM) of 8 K/V tiles at d = 128; odd
    GQA group sizes."""
    _check(ai.AttnShape(2, Hq, Hkv, 1000, 1000, 128, "bf16", causal), oracle_mod, 82, Hq * 10 + int(causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("Nq,Nk,causal", [(900, 900, True), (1000, 1000, False), (300, 2000, True),
                                          (130, 4500, False)])
def test_halves_ragged(attn, oracle_mod, dtype, Nq, Nk, causal):
    """Halves at d = 64: ragged rows and keys, Nq < Nk (bottom-right causal),
    tiles whose halves differ in length, one row past a tile."""
    _check(ai.AttnShape(1, 3, 3, Nq, Nk, 64, dtype, causal), oracle_mod, 84, Nq + Nk + int(causal))


@pytest.mark.parametrize("causal", [False, True])
def test_single_short_tiles(attn, oracle_mod, causal):
    """Few tiles of at most 3 K/V tiles: whole single tiles."""
    _check(ai.AttnShape(1, 4, 4, 384, 384, 64, "fp16", causal), oracle_mod, 85, int(causal))


def test_consecutive_pairs_odd_tiles(attn, oracle_mod):
    """Many items (more than one wave): consecutive pairs, with an odd tile
    count so the last item has one tile."""
    _check(ai.AttnShape(4, 41, 41, 2 * 128 + 7, 2 * 128 + 7, 64, "fp16", True), oracle_mod, 83)
