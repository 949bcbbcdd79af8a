"""The benchmark's multi-process path on CPU (gloo, world size 2).

The path partitions into independent replicas (no exchange step), so a run
on N GPUs is N ranks doing the same step, joined only by a barrier and a
max over ranks of the timed region; rank 0 prints the line.  These tests run
that logic as two gloo ranks: bench.py's own barrier, max-over-ranks and
whole-job aggregation, and its reference arm under torchrun."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    w, r, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.dist_barrier(w)
    # each rank "timed" a different total; the job is as slow as the slowest
    total_ms = 10.0 * (rank + 1)
    worst = bench.dist_max(w, total_ms, torch.device("cpu"))
    value = bench.job_value(w, 1e9, 4, worst)
    bench.dist_barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ws": w, "rank": r, "local": local, "worst": worst, "value": value}, f)
    torch.distributed.destroy_process_group()


def test_gloo_barrier_max_and_job_value(tmp_path):
    ws, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True, start_method="spawn")
    rows = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    for r, row in enumerate(rows):
        assert row["ws"] == 2 and row["rank"] == r and row["local"] == r
        assert row["worst"] == 20.0  # the max over ranks, seen by every rank
        # two replicas of 1 GFLOP x 4 steps in 20 ms: 0.4 TFLOP/s for the job
        assert row["value"] == pytest.approx(2 * 1e9 * 4 / 0.020 / 1e12)


def test_job_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_value(1, 2e12, 10, 1000.0) == pytest.approx(20.0)
    assert bench.job_value(4, 2e12, 10, 1000.0) == pytest.approx(80.0)


def test_reference_arm_under_torchrun():
    """Two ranks: rank 0 alone times the oracle and prints one line; rank 1
    exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "mha_n64", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["mha_n64", "paged_decode"])
def test_reference_line_contract(workload):
    """One process: the reference arm's JSON line carries every key of the
    benchmark contract, with the oracle described as the CPU baseline."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
           "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["higher_is_better"] is True
    assert line["dtype"] == "f64" and line["data"] == "synthetic" and line["vs_baseline"] is None
    assert line["config"]["workload"].startswith(workload)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["d2h_bytes_per_step"] == 0
