import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity against the stated bound (O max-abs 1e-3 for fp16 I/O, 8e-3 for
    bf16 I/O; LSE 1e-3): one line per benchmark configuration, then every
    other comparison that had an element over the stated bound, each such
    element with its oracle value.  ATTN_PARITY_REPORT=<path> also writes
    every record as JSON."""
    try:
        from tests import parity_util as pu
    except ImportError:
        return
    recs = pu.RECORDS
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity against the stated bound")
    tr.write_line(f"{'config / call':58s} {'dtype':5s} {'max|dO|':>9s} {'stated':>7s} {'over':>6s} {'of':>9s} "
                  f"{'ulps':>5s} {'max|dLSE|':>9s}  bound   (ulps: vs the rounded oracle, at |O| >= 1/16)")
    for r in recs:
        if not r["config"]:
            continue
        tr.write_line(f"{r['config'][:58]:58s} {r['dtype']:5s} {r['max_abs_O']:9.2e} {r['stated_tol_O']:7.0e} "
                      f"{r['n_over_stated']:6d} {r['n_elems']:9d} {r['ulps_to_rounded_oracle']:5.1f} "
                      f"{r.get('max_abs_LSE', float('nan')):9.2e}  {r['bound']}")
        for i, e, a in r["over_stated"]:
            tr.write_line(f"    element {i}: |dO| {e:.3e}, |O_oracle| {a:.3f}")
    others = [r for r in recs if not r["config"] and r["n_over_stated"] > 0]
    n_over = sum(r["n_over_stated"] for r in others)
    tr.write_line(f"other comparisons: {len(recs) - sum(1 for r in recs if r['config'])}; "
                  f"{len(others)} with elements over the stated bound ({n_over} elements):")
    for r in others:
        tr.write_line(f"  {r['test'][:70]} [{r['label'][:40]}] {r['dtype']} max|dO| {r['max_abs_O']:.2e}, "
                      f"{r['n_over_stated']} of {r['n_elems']} over")
        for i, e, a in r["over_stated"][:4]:
            tr.write_line(f"    element {i}: |dO| {e:.3e}, |O_oracle| {a:.3f}")
    path = os.environ.get("ATTN_PARITY_REPORT")
    if path:
        import json

        with open(path, "w") as f:
            json.dump(recs, f, indent=1)
