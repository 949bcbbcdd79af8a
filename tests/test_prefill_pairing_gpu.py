"""GPU parity of the prefill kernel's item pairings, through the C ABI,
against the fp64 oracle.  The host picks, per call: two heads of a GQA group
(even group sizes), one tile per item (every tile gets an SM), mirrored row
tiles (r, n-1-r) for a causal call in one wave, or consecutive row tiles.
Each case below is sized to land on one of them on a 152-SM GB300 (the
pairing changes only the schedule, never the result)."""
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
def test_mirror_pairs_causal(attn, oracle_mod, N):
    """5 heads x 31 or 32 row tiles: too many tiles for one per SM, but the
    mirrored pairs fit one wave; 31 tiles leave the middle tile alone."""
    _check(ai.AttnShape(1, 5, 5, N, N, 64, "fp16", True), oracle_mod, 80, N)


@pytest.mark.parametrize("window", [129, 700])
def test_mirror_pairs_window(attn, oracle_mod, window):
    _check(ai.AttnShape(1, 5, 5, 5000, 5000, 64, "bf16", True, window), oracle_mod, 81, window)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(3, 3), (6, 2)])
def test_single_tile_items(attn, oracle_mod, causal, Hq, Hkv):
    """Few tiles (every tile gets its own SM); odd GQA group sizes."""
    _check(ai.AttnShape(2, Hq, Hkv, 1000, 1000, 128, "bf16", causal), oracle_mod, 82, Hq * 10 + int(causal))


def test_consecutive_pairs_odd_tiles(attn, oracle_mod):
    """Many items (more than one wave): consecutive pairs, with an odd tile
    count so the last item has one tile."""
    _check(ai.AttnShape(4, 41, 41, 2 * 128 + 7, 2 * 128 + 7, 64, "fp16", True), oracle_mod, 83)
