"""FLOP / byte accounting pinned to the figures the pages print, and the
exact live-pair count checked against brute force."""
import json
import os

import pytest

from tiled_attention_forward_fwd_gb300 import accounting as acc
from tests import pins

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def close(a, b, rel):
    return abs(a - b) <= rel * abs(b)


def test_page_flops():
    f = G["attention_flops_per_layer"]
    assert close(acc.metric_flops(1, 1, f["N"], f["N"], f["d"], False), f["value"], f["rel_tol"])
    f = G["attention_flops_12_layers"]
    assert close(f["layers"] * acc.metric_flops(1, 1, f["N"], f["N"], f["d"], False), f["value"], f["rel_tol"])


def test_page_bytes():
    f = G["naive_score_bytes"]
    assert close(acc.naive_score_traffic_bytes(f["N"]) / 2 ** 20, f["value_mib"], f["rel_tol"])
    f = G["flash_bytes"]
    assert close(acc.flash_traffic_bytes_fp32(f["N"], f["d"], f["B_c"]) / 2 ** 20, f["value_mib"], f["rel_tol"])
    f = G["score_elements_32k"]
    assert close(f["s"] ** 2, f["value"], f["rel_tol"])


@pytest.mark.parametrize("Nq,Nk,causal,window", [(9, 9, False, 0), (9, 9, True, 0), (9, 9, True, 3),
                                                  (4, 9, True, 0), (4, 9, True, 2), (1, 9, True, 0),
                                                  (6, 4, True, 0), (17, 17, True, 1), (17, 17, True, 100)])
def test_live_pairs_brute_force(Nq, Nk, causal, window):
    brute = sum(pins.live(Nk - Nq + i, j, causal, window) for i in range(Nq) for j in range(Nk))
    assert acc.live_pairs_per_head(Nq, Nk, causal, window) == brute


def test_metric_convention():
    # square causal is half of full in the headline convention
    full = acc.metric_flops(2, 4, 4096, 4096, 64, False)
    assert acc.metric_flops(2, 4, 4096, 4096, 64, True) == full / 2
    assert full == 4 * 2 * 4 * 4096 * 4096 * 64
    # sliding window counts exact live pairs (W=4096 at N=8192)
    w = acc.metric_flops(4, 32, 8192, 8192, 128, True, 4096)
    assert w == 4 * 4 * 32 * 128 * (4096 * 4097 // 2 + 4096 * 4096)
    assert acc.compulsory_bytes(1, 2, 2, 64, 64, 64) == 2 * 64 * (2 * 128 + 2 * 128) + 4 * 128
