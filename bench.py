#!/usr/bin/env python
"""Benchmark: attention-forward TFLOP/s on one GB300 and the roofline fraction
of the dominant kernel, next to the fp64 CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass over every call of the workload with inputs resident in
HBM.  The default workload is the largest single-GPU configuration,
``long_prefill``: B=1, Hq=32, Hkv=8, N=32768, d=128, bf16, keys x3, causal
(8.8 TFLOP per step).  The step is captured once as a CUDA graph and
replayed; L2 is flushed between timed steps, outside the timed events: a
256 MiB write, then a 256 MiB read of another buffer, so that the timed step
starts with none of its inputs in L2 and with no dirty lines of the flush
left to write back.  Before the timed steps, after the warm-up steps,
untimed replays run for at least a second (the soak), so that the clocks
sampled during the timed region are those of a GPU under load.  Prints one
JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import attn_inputs as ai  # noqa: E402
from tiled_attention_forward_fwd_gb300 import accounting as acc  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_TEXT = {
    "mha_b2h4": "MHA forward B=2, H=4, d=64, fp16, N in {256,1024,4096} x causal in {true,false}",
    "mha_n64": "MHA forward B=1, H=2, N=64, d=64, fp16, causal in {false,true}",
    "gpt_stack": "12 causal layers B=8, H=12, N=2048, d=64, bf16, scale 1/8",
    "gqa_mqa": "B=4, Hq=32, Hkv in {8,1}, N=8192, d=128, bf16, causal; + window 4096",
    "long_prefill": "B=1, Hq=32, Hkv=8, N=32768, d=128, bf16, keys x3, causal",
    "mqa_decode": "decode B=4, Hq=32, Hkv in {1,8}, Nq=1, Nk=8192, d=128, bf16",
    "mha_n64_bw": "MHA forward B=512, H=32, N=64, d=64, fp16, causal in {false,true}",
    "paged_decode": "decode on a paged cache (16-token pages, shuffled pool), Hq=32, Hkv=8, Nq=1, d=128, bf16: "
                    "B=4 at 8192 tokens; B=32 at drawn lengths 512..8192",
    "mqa_decode_int8": "decode B=4, Hq=32, Hkv in {1,8}, Nq=1, Nk=8192, d=128, bf16 Q, int8 K/V (per-tensor scales)",
    "bwd_gpt_layer": "backward of a gpt_stack layer: B=8, H=12, N=2048, d=64, bf16, causal, scale 1/8",
    "bwd_gqa": "backward of B=4, Hq=32, Hkv=8, N=8192, d=128, bf16, causal",
    "paged_prefill": "chunked prefill on a paged cache (16-token pages, shuffled pool): B=4, Hq=32, Hkv=8, "
                     "Nq=2048 new rows per request, cache lengths drawn 2048..8192, d=128, bf16, causal",
    "mla_decode": "latent attention with absorbed queries, d_c=512, n_h=128, bf16, causal, scale 1/sqrt(128): "
                  "B=32, Nq=1, Nk=8192; B=8, Nq=4, Nk=8192",
}
# Device sources of each kernel family: a committed DRAM-traffic figure
# (profiles/traffic.json) counts only while they hash to the value recorded
# with it.  (Host launch code is not part of the key: an entry is re-taken
# whenever a path's launch configuration changes.)
KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd_sm103.cuh", "sm103_ptx.cuh", "fastdiv.h"],
    "attn_decode_kernel": ["attn_decode.cuh", "sm103_ptx.cuh"],
    "attn_short_kernel": ["attn_short.cuh", "sm103_ptx.cuh"],
    "attn_bwd_kernel": ["attn_bwd_sm103.cuh", "sm103_ptx.cuh"],
    "attn_mla_kernel": ["attn_mla.cuh", "attn_decode.cuh", "sm103_ptx.cuh"],
}


def metric_name(workload: str) -> str:
    if workload.startswith("bwd_"):
        return "attention bwd TFLOP/s (2.5x the forward's FLOPs)"
    return "attention fwd TFLOP/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_prefill", choices=ai.WORKLOAD_NAMES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--per-call", action="store_true", help="print per-call timings to stderr")
    ap.add_argument("--launch-floor", action="store_true",
                    help="only time empty-kernel CUDA graphs (the fixed cost of a launch) and print them")
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="untimed replays after the warm-up, before the timed steps")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing (weak scaling, no collective
# on the data path: every rank runs the same workload on its own GPU)
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def dist_barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def dist_max(ws, x: float, device) -> float:
    if ws <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(ws: int, flops_step: float, steps: int, max_total_ms: float) -> float:
    """Whole-job TFLOP/s of ws replicas (weak scaling: every rank runs the
    same step), each timed over `steps` steps, against the slowest rank."""
    return ws * flops_step * steps / (max_total_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- peaks, clocks, profiles
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, n in enumerate(names):
            if any(r[5 + i].lower() == "active" for r in self.rows):
                reasons.append(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the device sources of a kernel family ("attn_fwd_kernel", ...)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel.split("[")[0]]:
        with open(os.path.join(ROOT, "tiled_attention_forward_fwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, call_label: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, only if the
    kernel's sources are unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(call_label)
    if not e or e.get("kernel_src_sha") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- the workload on the GPU
def call_label(s) -> str:
    if isinstance(s, ai.PagedShape):
        return (f"paged_B{s.B}_Hq{s.Hq}_Hkv{s.Hkv}_Nq{s.Nq}_L{s.max_seq_len}_ps{s.page_size}_d{s.d}_{s.dtype}"
                f"_c{int(s.causal)}_w{s.window}")
    return (f"{'bwd_' if s.backward else ''}B{s.B}_Hq{s.Hq}_Hkv{s.Hkv}_Nq{s.Nq}_Nk{s.Nk}_d{s.d}_{s.dtype}"
            f"{'_kv8' if s.kv_int8 else ''}{'_mla' if s.mla else ''}_c{int(s.causal)}_w{s.window}")


def prepare_paged(shape, cid, layer, device):
    """One call on a paged cache: seeded pools, table and lengths."""
    import tiled_attention_forward_fwd_gb300 as attn

    q, k, v, table, lens = ai.make_paged(shape, cid, layer)
    host = {"q": q, "k": k, "v": v, "table": table, "lens": lens}
    c = {"shape": shape, "paged": True, **{n + "_host": t for n, t in host.items()},
         **{n: t.to(device) for n, t in host.items()}}
    c["o"] = torch.empty_like(c["q"])
    c["lse"] = torch.empty((shape.B, shape.Hq, shape.Nq), device=device, dtype=torch.float32)
    c["dtype_code"] = attn.ATTN_DTYPE_BF16 if shape.dtype == "bf16" else attn.ATTN_DTYPE_FP16
    lens_l = lens.tolist()
    c["flops"] = acc.paged_flops(shape, lens_l)
    c["bytes"] = acc.paged_bytes(shape, lens_l)
    c["label"] = call_label(shape)
    wsb = attn.attn_fwd_paged_workspace_bytes(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.max_seq_len, shape.d)
    c["ws"] = torch.empty(wsb, dtype=torch.uint8, device=device)
    path = attn.attn_fwd_paged_path(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.max_seq_len, shape.d)
    c["path"] = path
    c["kernel"] = "attn_fwd_kernel[paged]" if path == attn.ATTN_PATH_PREFILL else "attn_decode_kernel[paged]"
    c["launches"] = 2 if path == attn.ATTN_PATH_SPLIT_KV else 1
    return c


def prepare_bwd(shape, cid, layer, device):
    """One backward call: seeded Q, K, V and upstream gradient; O and LSE
    from the library's forward (computed here, before any timing)."""
    import tiled_attention_forward_fwd_gb300 as attn

    q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
    do = ai.normal_tensor(ai.seed_for(cid, layer, "G"), tuple(q.shape), shape.dtype)
    c = {"shape": shape, "backward": True, "q_host": q, "k_host": k, "v_host": v, "do_host": do,
         "q": q.to(device), "k": k.to(device), "v": v.to(device), "do": do.to(device)}
    c["o"], c["lse"] = attn.flash_attn_forward(c["q"], c["k"], c["v"], causal=shape.causal, window=shape.window,
                                               sm_scale=shape.scale)
    torch.cuda.synchronize(device)
    c["o_host"], c["lse_host"] = c["o"].cpu(), c["lse"].cpu()
    c["dq"], c["dk"], c["dv"] = torch.empty_like(c["q"]), torch.empty_like(c["k"]), torch.empty_like(c["v"])
    c["dtype_code"] = attn.ATTN_DTYPE_BF16 if shape.dtype == "bf16" else attn.ATTN_DTYPE_FP16
    c["flops"] = acc.shape_flops(shape)
    c["bytes"] = acc.shape_bytes(shape)
    c["label"] = call_label(shape)
    c["ws"] = torch.empty(attn.attn_bwd_workspace_bytes(shape.B, shape.Hq, shape.Nq, shape.d), dtype=torch.uint8,
                          device=device)
    c["path"] = None
    c["kernel"] = "attn_bwd_kernel"
    c["launches"] = 3  # D and the accumulator, the gradients, dQ
    return c


def prepare_mla(shape, cid, layer, device):
    """One latent-attention call: absorbed queries (B, n_h, Nq, 512) and the
    latent cache (B, Nk, 512), drawn as Q and the single K/V head."""
    import tiled_attention_forward_fwd_gb300 as attn

    q, k, _ = ai.make_qkv(shape, config_id=cid, layer=layer)
    c = {"shape": shape, "mla": True, "q_host": q, "c_host": k[:, 0].contiguous(), "q": q.to(device)}
    c["c"] = c["c_host"].to(device)
    c["o"] = torch.empty_like(c["q"])
    c["lse"] = torch.empty((shape.B, shape.Hq, shape.Nq), device=device, dtype=torch.float32)
    c["dtype_code"] = attn.ATTN_DTYPE_BF16 if shape.dtype == "bf16" else attn.ATTN_DTYPE_FP16
    c["flops"] = acc.shape_flops(shape)
    c["bytes"] = acc.shape_bytes(shape)
    c["label"] = call_label(shape)
    c["ws"] = torch.empty(attn.attn_fwd_mla_workspace_bytes(shape.B, shape.Hq, shape.Nq, shape.Nk, shape.d),
                          dtype=torch.uint8, device=device)
    c["path"] = None
    c["kernel"] = "attn_mla_kernel"
    c["launches"] = 2  # the split kernel, the merge
    return c


def prepare(workload: str, device):
    import tiled_attention_forward_fwd_gb300 as attn

    calls = []
    for shape, cid, layer in ai.workload_calls(workload):
        if isinstance(shape, ai.PagedShape):
            calls.append(prepare_paged(shape, cid, layer, device))
            continue
        if shape.backward:
            calls.append(prepare_bwd(shape, cid, layer, device))
            continue
        if shape.mla:
            calls.append(prepare_mla(shape, cid, layer, device))
            continue
        if shape.kv_int8:
            q, k, ks, v, vs = ai.make_qkv_int8(shape, cid, layer)
        else:
            q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
        c = {"shape": shape, "q_host": q, "k_host": k, "v_host": v,
             "q": q.to(device), "k": k.to(device), "v": v.to(device)}
        if shape.kv_int8:
            c["k_scale"], c["v_scale"] = ks, vs
        c["o"] = torch.empty_like(c["q"])
        c["lse"] = torch.empty((shape.B, shape.Hq, shape.Nq), device=device, dtype=torch.float32)
        c["dtype_code"] = attn.ATTN_DTYPE_BF16 if shape.dtype == "bf16" else attn.ATTN_DTYPE_FP16
        c["flops"] = acc.shape_flops(shape)
        c["bytes"] = acc.shape_bytes(shape)
        c["label"] = call_label(shape)
        # split paths (split-KV decode for few query rows, stream-K split of a
        # prefill that fills less than two waves): caller-provided workspace
        wsb = attn.attn_fwd_workspace_bytes(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d)
        path = attn.attn_fwd_path(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d, wsb > 0)
        if path == attn.ATTN_PATH_PREFILL_SPLIT and shape.window > 0:
            path = attn.ATTN_PATH_PREFILL  # the split is not used with a window
        split = path in (attn.ATTN_PATH_SPLIT_KV, attn.ATTN_PATH_SPLIT_KV_FUSED, attn.ATTN_PATH_PREFILL_SPLIT)
        if shape.kv_int8:  # the int8 entry plans its chunks for its own kernel
            wsb = attn.attn_fwd_kv_int8_workspace_bytes(shape.B, shape.Hq, shape.Hkv, shape.Nq, shape.Nk, shape.d)
        c["ws"] = torch.empty(wsb, dtype=torch.uint8, device=device) if split else None
        c["path"] = path
        c["kernel"] = {attn.ATTN_PATH_PREFILL: "attn_fwd_kernel", attn.ATTN_PATH_PREFILL_SPLIT: "attn_fwd_kernel",
                       attn.ATTN_PATH_SPLIT_KV: "attn_decode_kernel", attn.ATTN_PATH_SPLIT_KV_FUSED: "attn_decode_kernel",
                       attn.ATTN_PATH_SHORT: "attn_short_kernel"}[path]
        c["launches"] = 2 if path == attn.ATTN_PATH_SPLIT_KV else 1  # split kernel + merge kernel
        calls.append(c)
    return calls


def launch(c, stream_handle):
    import tiled_attention_forward_fwd_gb300 as attn

    s = c["shape"]
    ws = c["ws"]
    if c.get("backward"):
        st = attn.attn_bwd(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["o"].data_ptr(),
                           c["do"].data_ptr(), c["lse"].data_ptr(), c["dq"].data_ptr(), c["dk"].data_ptr(),
                           c["dv"].data_ptr(), s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, s.causal, s.window, s.scale,
                           c["dtype_code"], ws.data_ptr(), ws.numel(), stream_handle)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_bwd failed: {attn.attn_status_string(st)}")
        return
    if c.get("paged"):
        st = attn.attn_fwd_paged(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["table"].data_ptr(),
                                 c["lens"].data_ptr(), c["o"].data_ptr(), c["lse"].data_ptr(), s.B, s.Hq, s.Hkv,
                                 s.Nq, s.max_seq_len, s.d, s.page_size, c["k"].shape[0], c["table"].shape[1],
                                 s.causal, s.window, s.scale, c["dtype_code"], ws.data_ptr(), ws.numel(),
                                 stream_handle)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_fwd_paged failed: {attn.attn_status_string(st)}")
        return
    if c.get("mla"):
        st = attn.attn_fwd_mla(c["q"].data_ptr(), c["c"].data_ptr(), c["o"].data_ptr(), c["lse"].data_ptr(), s.B,
                               s.Hq, s.Nq, s.Nk, s.d, s.causal, s.window, s.scale, c["dtype_code"], ws.data_ptr(),
                               ws.numel(), stream_handle)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_fwd_mla failed: {attn.attn_status_string(st)}")
        return
    if s.kv_int8:
        st = attn.attn_fwd_kv_int8(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["k_scale"],
                                   c["v_scale"], c["o"].data_ptr(), c["lse"].data_ptr(), s.B, s.Hq, s.Hkv, s.Nq,
                                   s.Nk, s.d, s.causal, s.window, s.scale, c["dtype_code"], ws.data_ptr(),
                                   ws.numel(), stream_handle)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_fwd_kv_int8 failed: {attn.attn_status_string(st)}")
        return
    st = attn.attn_fwd_ex(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["o"].data_ptr(),
                          c["lse"].data_ptr(), s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, s.causal, s.window, s.scale,
                          c["dtype_code"], None if ws is None else ws.data_ptr(),
                          0 if ws is None else ws.numel(), stream_handle)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"attn_fwd_ex failed: {attn.attn_status_string(st)}")


def make_event():
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


def build_graph(calls, stream, per_call_events: bool):
    """Capture one step (every call, back to back).  With per_call_events a
    timing event sits between launches; that graph gives the per-call times,
    but an event between two kernels also keeps the second from starting its
    prologue early (programmatic dependent launch), so the step time comes
    from the graph without them."""
    evs = [make_event() for _ in range(len(calls) + 1)] if per_call_events else []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        # warm the launch path (tensor-map encoder, kernel attributes) before capture
        for c in calls:
            launch(c, stream.cuda_stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            if per_call_events:
                evs[0].record(stream)
            for i, c in enumerate(calls):
                launch(c, stream.cuda_stream)
                if per_call_events:
                    evs[i + 1].record(stream)
    return g, evs


def device_timing(calls, steps, warmup, device, stream, soak_s=1.0):
    import tiled_attention_forward_fwd_gb300 as attn

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    flush_rd = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def flush_l2():
        flush.fill_(1.0)  # evicts everything (larger than the 129 MB L2) ...
        flush_rd.sum()    # ... and this read leaves only clean lines behind

    g, _ = build_graph(calls, stream, per_call_events=False)
    g_calls, evs = build_graph(calls, stream, per_call_events=True)
    t_start, t_stop = make_event(), make_event()
    for _ in range(warmup):
        with torch.cuda.stream(stream):
            flush_l2()
            g.replay()
            flush_l2()
            g_calls.replay()
    torch.cuda.synchronize(device)
    soak = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < soak_s:
        with torch.cuda.stream(stream):
            for _ in range(4):
                flush_l2()
                g.replay()
                soak += 1
        stream.synchronize()
    step_ms, call_ms = [], [[] for _ in calls]
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush_l2()
            t_start.record(stream)
            g.replay()
            t_stop.record(stream)
        stream.synchronize()
        step_ms.append(t_start.elapsed_time(t_stop))
    # per-call device times (the roofline's dominant call), same flush
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush_l2()
            g_calls.replay()
        stream.synchronize()
        for i in range(len(calls)):
            call_ms[i].append(evs[i].elapsed_time(evs[i + 1]))
    st = attn.attn_device_status(stream.cuda_stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel status after timing: {attn.attn_status_string(st)}")
    return step_ms, call_ms, soak


def e2e_timing(calls, steps, warmup, device, stream):
    """Same metric through the public C entry on HOST buffers: every step copies
    each call's Q, K, V from pinned host memory, runs, and copies O and LSE
    back."""
    import tiled_attention_forward_fwd_gb300 as attn

    pinned = []
    need = 0
    for c in calls:
        s = c["shape"]
        if c.get("backward"):
            # Q, K, V, O, dO and LSE copied in; dQ, dK, dV copied back
            ph = {k: c[k + "_host"].pin_memory() for k in ("q", "k", "v", "o", "do", "lse")}
            for k in ("dq", "dk", "dv"):
                ph[k] = torch.empty(c[k].shape, dtype=c[k].dtype).pin_memory()
            pinned.append(ph)
            continue
        if c.get("paged") or c.get("mla") or s.kv_int8:
            # the inputs of a paged call (pools, table, lengths, Q), of a
            # latent call (Q, latent cache) or of an int8 call (Q, codes) are
            # copied into its device tensors, then the call runs on them
            names = ("q", "k", "v")
            if c.get("paged"):
                names = ("q", "k", "v", "table", "lens")
            elif c.get("mla"):
                names = ("q", "c")
            ph = {k: c[k + "_host"].pin_memory() for k in names}
            ph["o"] = torch.empty_like(ph["q"]).pin_memory()
            ph["lse"] = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32).pin_memory()
            pinned.append(ph)
            continue
        ph = {k: c[k + "_host"].pin_memory() for k in ("q", "k", "v")}
        ph["o"] = torch.empty_like(ph["q"]).pin_memory()
        ph["lse"] = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32).pin_memory()
        pinned.append(ph)
        need = max(need, attn.attn_fwd_host_staging_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, 1))
    buf = torch.empty(need + 256, dtype=torch.uint8, device=device)
    base = (buf.data_ptr() + 255) & ~255
    h2d = d2h = 0
    for c in calls:
        s = c["shape"]
        if c.get("backward"):
            h2d += (2 * c["q"].numel() + c["k"].numel() + c["v"].numel() + c["do"].numel()) * 2 + c["lse"].numel() * 4
            d2h += (c["dq"].numel() + c["dk"].numel() + c["dv"].numel()) * 2
            continue
        if c.get("mla"):
            h2d += (c["q"].numel() + c["c"].numel()) * 2
            d2h += c["o"].numel() * 2 + s.B * s.Hq * s.Nq * 4
            continue
        h2d += c["q"].numel() * 2 + (c["k"].numel() + c["v"].numel()) * c["k"].element_size()
        if c.get("paged"):
            h2d += (c["table"].numel() + c["lens"].numel()) * 4
        d2h += c["o"].numel() * 2 + s.B * s.Hq * s.Nq * 4

    def one_step():
        for c, ph in zip(calls, pinned):
            s = c["shape"]
            if c.get("backward"):
                with torch.cuda.stream(stream):
                    for k in ("q", "k", "v", "o", "do", "lse"):
                        c[k].copy_(ph[k], non_blocking=True)
                    launch(c, stream.cuda_stream)
                    for k in ("dq", "dk", "dv"):
                        ph[k].copy_(c[k], non_blocking=True)
                continue
            if c.get("paged") or c.get("mla") or s.kv_int8:
                names = ("q", "k", "v", "table", "lens") if c.get("paged") else ("q", "c") if c.get("mla") \
                    else ("q", "k", "v")
                with torch.cuda.stream(stream):
                    for k in names:
                        c[k].copy_(ph[k], non_blocking=True)
                    launch(c, stream.cuda_stream)
                    ph["o"].copy_(c["o"], non_blocking=True)
                    ph["lse"].copy_(c["lse"], non_blocking=True)
                continue
            st = attn.attn_fwd_host(ph["q"].data_ptr(), ph["k"].data_ptr(), ph["v"].data_ptr(), ph["o"].data_ptr(),
                                    ph["lse"].data_ptr(), s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, s.causal, s.window,
                                    s.scale, c["dtype_code"], base, need, stream.cuda_stream)
            if st != attn.ATTN_OK:
                raise RuntimeError(f"attn_fwd_host failed: {attn.attn_status_string(st)}")

    for _ in range(warmup):
        one_step()
    stream.synchronize()
    t0, t1 = make_event(), make_event()
    t0.record(stream)
    for _ in range(steps):
        one_step()
    t1.record(stream)
    stream.synchronize()
    ms = t0.elapsed_time(t1) / steps
    # result check on the last step: what was copied back equals the device tensors
    for c, ph in zip(calls, pinned):
        for k in (("dq", "dk", "dv") if c.get("backward") else ("o",)):
            if not torch.equal(ph[k], c[k].cpu()):
                raise RuntimeError("host-buffer path disagrees with the device path")
    return ms, h2d, d2h


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)
def oracle_sample(workload: str, budget_s: float, seed: int = 0, nthreads: int = 0):
    """Time the fp64 oracle on a bounded, seeded sample of the workload's
    query rows (every call contributes).  nthreads = 0: all cores (OpenMP);
    a positive count is used by the plain forward calls.  Returns
    (flops_done, seconds, cores, description)."""
    import oracle

    oracle.build()
    cores = oracle.max_threads()
    calls = ai.workload_calls(workload)
    rng = np.random.default_rng(seed)
    prepared = []
    for shape, cid, layer in calls:
        if isinstance(shape, ai.PagedShape):
            q, k, v, table, lens = ai.make_paged(shape, cid, layer)
            prepared.append((shape, q, k.to(torch.float64), v.to(torch.float64), table, lens))
            continue
        if shape.backward:
            q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
            do = ai.normal_tensor(ai.seed_for(cid, layer, "G"), tuple(q.shape), shape.dtype)
            prepared.append((shape, q, k, v, do, "bwd"))
            continue
        if shape.kv_int8:  # the oracle reads the exactly dequantised cache
            q, kc, ks, vc, vs = ai.make_qkv_int8(shape, cid, layer)
            k, v = kc.to(torch.float64) * ks, vc.to(torch.float64) * vs
        else:
            q, k, v = ai.make_qkv(shape, config_id=cid, layer=layer)
            if shape.mla:  # the latent cache serves as keys and values
                v = k
        prepared.append((shape, q.reshape(-1, shape.d), k.to(torch.float64), v.to(torch.float64)))

    def run_paged(shape, q, k, v, table, lens, rows_per_call):
        # whole requests (all heads and rows), as many as the row budget covers
        n = min(shape.B, max(1, rows_per_call // (shape.Hq * shape.Nq)))
        covered.append(n == shape.B)
        ids = np.sort(rng.choice(shape.B, size=n, replace=False))
        sel = torch.from_numpy(ids)
        t0 = time.perf_counter()
        oracle.attention_paged(q[sel], k, v, table[sel], lens[sel], shape.causal, shape.window, shape.scale)
        return acc.paged_flops(shape, lens[sel].tolist()), time.perf_counter() - t0

    covered = []  # per call of the last run: the whole call was sampled

    def run_bwd(shape, q, k, v, do, rows_per_call):
        # the oracle's gradients of a self-contained piece of the call: batch
        # 0, the first GQA group, the first n positions (a causal prefix
        # sees only itself; non-causal: its own keys)
        g = shape.Hq // shape.Hkv
        n = max(1, min(shape.Nq, rows_per_call // g))
        covered.append(n == shape.Nq and shape.B == 1 and shape.Hkv == 1)
        sub = ai.AttnShape(1, g, 1, n, n, shape.d, shape.dtype, shape.causal, shape.window, shape.sm_scale,
                           backward=True)
        t0 = time.perf_counter()
        oracle.attention_bwd(q[:1, :g, :n], k[:1, :1, :n], v[:1, :1, :n], do[:1, :g, :n], causal=shape.causal,
                             window=shape.window, sm_scale=shape.scale)
        return acc.shape_flops(sub, exact=True), time.perf_counter() - t0

    def run(rows_per_call):
        flops = 0.0
        t = 0.0
        covered.clear()
        for shape, *tensors in prepared:
            if tensors and isinstance(tensors[-1], str):
                f, dt = run_bwd(shape, *tensors[:-1], rows_per_call)
                flops += f
                t += dt
                continue
            if isinstance(shape, ai.PagedShape):
                f, dt = run_paged(shape, *tensors, rows_per_call)
                flops += f
                t += dt
                continue
            qf, kf, vf = tensors
            total = shape.B * shape.Hq * shape.Nq
            n = min(total, rows_per_call)
            covered.append(n == total)
            ids = np.sort(rng.choice(total, size=n, replace=False)).astype(np.int64)
            i = ids % shape.Nq
            pos = shape.Nk - shape.Nq + i
            if shape.causal:
                live = np.minimum(pos + 1, shape.window if shape.window > 0 else pos + 1)
            else:
                live = np.full_like(i, shape.Nk)
            flops += 4.0 * shape.d * float(live.sum())
            qr = qf[torch.from_numpy(ids)]
            t0 = time.perf_counter()
            oracle.attention_rows(qr, ids, kf, vf, B=shape.B, Hq=shape.Hq, Nq=shape.Nq, causal=shape.causal,
                                  window=shape.window, sm_scale=shape.scale, nthreads=nthreads)
            t += time.perf_counter() - t0
        return flops, t

    rows = 16
    run(rows)  # untimed: OpenMP start-up and first touch of the oracle's scratch
    f, t = run(rows)
    while t < budget_s / 8 and rows < 1 << 22 and not all(covered):
        rows *= 4
        f, t = run(rows)
    if t < budget_s / 2 and not all(covered):
        scale = max(1.0, (budget_s * 0.75) / max(t, 1e-6))
        rows = int(rows * scale)
        f, t = run(rows)
    if all(covered):
        desc = (f"every query row of every call in {workload} (the whole workload fits the sample), "
                f"fp64 oracle on {cores} OpenMP threads; work = 4*d per live pair")
    else:
        desc = (f"{rows} seeded random query rows per call of every call in {workload} "
                f"(capped at the call's rows; paged calls: whole requests covering that many rows), "
                f"fp64 oracle on {cores} OpenMP threads; work = 4*d per live pair")
    return f, t, cores, desc


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    cid = ai.workload_calls(args.workload)
    per_step_budget = max(0.5, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, per_step_budget / 4)
    flops = secs = 0.0
    cores, desc = 0, ""
    for k in range(args.steps):
        f, t, cores, desc = oracle_sample(args.workload, per_step_budget, seed=k + 1)
        flops += f
        secs += t
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": metric_name(args.workload), "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                   "sample": "bounded row sample per step (oracle is row-independent)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- main
def launch_floor(device) -> dict:
    """Device time, between two events captured around it in a CUDA graph (as
    bench.py times one call), of one empty kernel launched like the
    library's kernels, for a few grid / shared-memory sizes, and of two of
    them back to back: the fixed cost that a call of one or two launches
    cannot go below."""
    import tiled_attention_forward_fwd_gb300 as attn

    stream = torch.cuda.Stream(device)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    out = {}
    for grid, smem, n in ((1, 0, 1), (152, 0, 1), (608, 0, 1), (152, 200 * 1024, 1), (608, 100 * 1024, 1),
                          (608, 100 * 1024, 2)):
        e0, e1 = make_event(), make_event()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e0.record(torch.cuda.current_stream())
            for _ in range(n):
                st = attn.attn_empty_launch(grid, 160, smem, torch.cuda.current_stream().cuda_stream)
                if st != attn.ATTN_OK:
                    raise RuntimeError(attn.attn_status_string(st))
            e1.record(torch.cuda.current_stream())
        times = []
        for k in range(60):
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
                g.replay()
            stream.synchronize()
            if k >= 10:
                times.append(e0.elapsed_time(e1) * 1e3)
        out[f"grid{grid}_smem{smem // 1024}KB_x{n}"] = float(np.median(times))
    return out


def main():
    args = parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    if args.launch_floor:
        device = torch.device("cuda", 0)
        torch.cuda.set_device(device)
        print(json.dumps({"launch_floor_us_per_graph": launch_floor(device),
                          "note": "median device time between events around empty kernels inside a CUDA graph (160 threads each), as bench.py times a call"}), flush=True)
        return 0
    ws, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(ws, "nccl")
    import tiled_attention_forward_fwd_gb300 as attn

    attn.lib()
    peaks, peaks_src = load_peaks()
    calls = prepare(args.workload, device)
    stream = torch.cuda.Stream(device)
    steps, warmup = args.steps, max(3, args.warmup)

    dist_barrier(ws)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(local)
    sampler.start()
    step_ms, call_ms, soak_steps = device_timing(calls, steps, warmup, device, stream, args.soak_seconds)
    clocks = sampler.stop()
    torch.cuda.synchronize(device)
    dist_barrier(ws)

    total_ms = dist_max(ws, float(sum(step_ms)), device)
    flops_step = sum(c["flops"] for c in calls)
    value = job_value(ws, flops_step, steps, total_ms)
    ms_per_step = total_ms / steps

    # dominant kernel: the call with the largest share of device time
    avg = [float(np.mean(m)) for m in call_ms]
    dom = int(np.argmax(avg))
    dc = calls[dom]
    s = dc["shape"]
    ai_flop_per_byte = dc["flops"] / dc["bytes"]
    peak_t = peaks["bf16_tflops"]
    ridge = peak_t * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if ai_flop_per_byte >= ridge:
        achieved = dc["flops"] / (avg[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                "frac": achieved / peak_t}
        if "bf16_tflops_sustained" in peaks:  # context: the power-capped rate of a seconds-long GEMM loop
            roof["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    else:
        achieved = dc["bytes"] / (avg[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    roof["traffic"] = profiled_traffic(args.workload, dc["label"], dc["kernel"])
    roof["kernel"] = f"{dc['kernel']}<{s.d},{'bf16' if s.dtype == 'bf16' else 'fp16'}> {dc['label']}"
    roof["algorithmic"] = {"flops": dc["flops"], "bytes": dc["bytes"]}
    roof["peak_source"] = f"{peaks_src} (burst bf16 dense; fp16 same rate)" if roof["bound"] == "tensor" \
        else f"{peaks_src} HBM copy"
    roof["launch_ms"] = avg[dom]

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_timing(calls, max(3, steps // 4), 2, device, stream)
        e2e_ms = dist_max(ws, e2e_ms, device)
        e2e = {"value": ws * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        f, t, cores, desc = oracle_sample(args.workload, args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": t}
        if args.workload in ("mha_n64", "mha_b2h4", "mha_n64_bw"):
            # the small configurations: the same oracle on one core as well
            f1, t1, _, _ = oracle_sample(args.workload, min(4.0, args.cpu_seconds / 3), seed=1, nthreads=1)
            cpu["one_core_value"] = f1 / t1 / 1e12

    if args.per_call and rank == 0:
        for c, a in zip(calls, avg):
            print(f"{c['label']}: {a * 1e3:.1f} us  {c['flops'] / (a * 1e-3) / 1e12:.1f} TFLOP/s  "
                  f"{c['bytes'] / (a * 1e-3) / 1e9:.0f} GB/s", file=sys.stderr)

    if rank == 0:
        line = {
            "metric": metric_name(args.workload), "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": steps,
            "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": calls[0]["shape"].dtype, "data": "synthetic",
            "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                       "calls_per_step": len(calls),
                       "flop_convention": "4*B*Hq*N^2*d, halved for square causal; exact live pairs otherwise",
                       "l2": "flushed between timed steps outside the timed events: 256 MiB write, then 256 MiB read",
                       "launch": "one CUDA graph per step (per-call times from a second graph with events between calls)",
                       "soak_steps": soak_steps,
                       "parallelism": f"replicas x{ws}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": steps * sum(c["launches"] for c in calls), "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
