"""Seeded synthetic inputs for attention, shared by the CUDA path's tests/bench
and by the CPU oracle.

This module holds no attention arithmetic: it only draws numbers.  The
workloads use Q, K, V drawn i.i.d. from N(0, 1) (optionally scaled, e.g. keys
x3 for the long-context stress case) and rounded to fp16 or bf16.

Generator (counter-based, so any element can be drawn independently and the
x86 and aarch64 hosts agree):

* splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): output n of stream ``seed`` is
  ``mix64(seed + (n + 1) * 0x9E3779B97F4A7C15)`` with the published finaliser
  ``mix64``.
* 53-bit uniforms in the open interval (0, 1): ``((x >> 11) + 0.5) * 2**-53``.
* Box-Muller (Box & Muller, 1958): element pair (2k, 2k+1) takes uniforms
  u1 = U(2k), u2 = U(2k+1) and gives r*cos(2*pi*u2), r*sin(2*pi*u2) with
  r = sqrt(-2 ln u1).
* The float64 normal times ``scale`` is rounded once (round-to-nearest-even)
  to the storage dtype by torch's CPU conversion.

Seeds follow ``seed = 1000 * config_id + 10 * layer + {0: Q, 1: K, 2: V}``.
"""
from __future__ import annotations

import hashlib
import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # pairs per chunk (bounds temporaries to ~32 MB each)

GENERATOR_VERSION = "splitmix64-boxmuller-v1"

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the splitmix64 stream ``seed``."""
    n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + n * GAMMA)


def uniform53(x: np.ndarray) -> np.ndarray:
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def _fill_chunk(out: np.ndarray, seed: int, numel: int, p0: int, p1: int) -> None:
    u = uniform53(splitmix64(seed, 2 * p0, 2 * (p1 - p0)))
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = (2.0 * math.pi) * u2
    pair = np.empty(2 * (p1 - p0), dtype=np.float64)
    pair[0::2] = r * np.cos(t)
    pair[1::2] = r * np.sin(t)
    e0, e1 = 2 * p0, min(numel, 2 * p1)
    out[e0:e1] = pair[: e1 - e0]


def normal_f64(seed: int, numel: int) -> np.ndarray:
    """``numel`` i.i.d. N(0,1) float64 values of stream ``seed``.

    Chunks are independent (counter-based), so they are filled by a thread
    pool; the result does not depend on the number of threads."""
    out = np.empty(numel, dtype=np.float64)
    npairs = (numel + 1) // 2
    starts = list(range(0, npairs, _CHUNK))
    if len(starts) <= 1:
        for p0 in starts:
            _fill_chunk(out, seed, numel, p0, min(npairs, p0 + _CHUNK))
        return out
    workers = min(len(starts), os.cpu_count() or 1, 32)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda p0: _fill_chunk(out, seed, numel, p0, min(npairs, p0 + _CHUNK)), starts))
    return out


def normal_tensor(seed: int, shape, dtype: str, scale: float = 1.0) -> torch.Tensor:
    """A CPU tensor of ``shape`` drawn from stream ``seed``, times ``scale``,
    rounded once to ``dtype`` ("fp16" | "bf16" | "f64")."""
    numel = int(np.prod(shape)) if len(shape) else 1
    z = normal_f64(seed, numel)
    if scale != 1.0:
        z = z * scale
    t = torch.from_numpy(z).reshape(tuple(shape))
    if dtype == "f64":
        return t
    return t.to(DTYPES[dtype])


def seed_for(config_id: int, layer: int, which: str) -> int:
    return 1000 * config_id + 10 * layer + {"Q": 0, "K": 1, "V": 2, "L": 3, "P": 4, "G": 5}[which]


@dataclass(frozen=True)
class AttnShape:
    """One attention call: Q,O (B,Hq,Nq,d); K,V (B,Hkv,Nk,d)."""

    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    dtype: str = "fp16"
    causal: bool = False
    window: int = 0
    sm_scale: float | None = None
    key_scale: float = 1.0
    kv_int8: bool = False  # K and V stored as int8 codes with one scale per tensor
    backward: bool = False  # the call is the backward pass of this forward
    mla: bool = False  # latent attention: Hkv = 1, d = d_c, K = V = the latent cache, Q the absorbed queries

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(self.d)


def make_qkv_int8(shape: AttnShape, config_id: int = 0, layer: int = 0):
    """Seeded (Q, K codes, K scale, V codes, V scale): Q in the storage
    dtype; K and V drawn like make_qkv's (before rounding) and quantised per tensor
    (quantize_int8)."""
    q = normal_tensor(seed_for(config_id, layer, "Q"), (shape.B, shape.Hq, shape.Nq, shape.d), shape.dtype)
    k = normal_tensor(seed_for(config_id, layer, "K"), (shape.B, shape.Hkv, shape.Nk, shape.d), "f64",
                      scale=shape.key_scale)
    v = normal_tensor(seed_for(config_id, layer, "V"), (shape.B, shape.Hkv, shape.Nk, shape.d), "f64")
    kc, ks = quantize_int8(k)
    vc, vs = quantize_int8(v)
    return q, kc, ks, vc, vs


def make_qkv(shape: AttnShape, config_id: int = 0, layer: int = 0):
    """Seeded (Q, K, V) CPU tensors in the storage dtype, contiguous."""
    q = normal_tensor(seed_for(config_id, layer, "Q"), (shape.B, shape.Hq, shape.Nq, shape.d), shape.dtype)
    k = normal_tensor(seed_for(config_id, layer, "K"), (shape.B, shape.Hkv, shape.Nk, shape.d), shape.dtype,
                      scale=shape.key_scale)
    v = normal_tensor(seed_for(config_id, layer, "V"), (shape.B, shape.Hkv, shape.Nk, shape.d), shape.dtype)
    return q, k, v


@dataclass(frozen=True)
class PagedShape:
    """One call on a paged K/V cache: Q,O (B,Hq,Nq,d); K,V pools
    (num_pages,Hkv,page_size,d); a page table (B,max_pages) and a length per
    request.  ``lens`` fixes the lengths; otherwise they are drawn uniformly
    from [min_len, max_seq_len]."""

    B: int
    Hq: int
    Hkv: int
    Nq: int
    max_seq_len: int
    d: int
    page_size: int = 16
    dtype: str = "bf16"
    causal: bool = True
    window: int = 0
    sm_scale: float | None = None
    lens: tuple | None = None
    min_len: int = 1
    spare_pages: int = 0  # pool pages no request owns

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def max_pages(self) -> int:
        return -(-self.max_seq_len // self.page_size)


def _uniform_ints(seed: int, n: int, lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """n integers, the k-th uniform on [lo_k, hi_k] (floor of a 53-bit uniform)."""
    u = uniform53(splitmix64(seed, 0, n))
    return (lo + np.floor(u * (hi - lo + 1)).astype(np.int64)).astype(np.int64)


def make_paged(shape: PagedShape, config_id: int = 0, layer: int = 0, poison: bool = True):
    """Seeded paged inputs: ``(q, k_pool, v_pool, block_table, seq_lens)`` as
    CPU tensors (int32 for the table and lengths).

    Each request gets ceil(len / page_size) pages.  The pool is shuffled
    (Fisher-Yates, Knuth TAOCP vol. 2, Algorithm 3.4.2P, driven by the
    stream above), so a request's pages are scattered, as in a fragmented
    cache.  Table entries past a request's pages are -1.  With ``poison``,
    every pool slot that no request owns (spare pages, and slots past a
    request's length in its last page) holds NaN, so that any read of one
    shows in the result."""
    B, ps = shape.B, shape.page_size
    if shape.lens is not None:
        lens = np.asarray(shape.lens, dtype=np.int64)
        if lens.shape != (B,):
            raise ValueError("lens must have one entry per request")
    else:
        lens = _uniform_ints(seed_for(config_id, layer, "L"), B, np.full(B, shape.min_len),
                             np.full(B, shape.max_seq_len))
    pages = -(-lens // ps)
    num_pages = int(pages.sum()) + shape.spare_pages
    perm = np.arange(num_pages, dtype=np.int64)
    if num_pages > 1:
        idx = np.arange(num_pages - 1, 0, -1)
        js = _uniform_ints(seed_for(config_id, layer, "P"), num_pages - 1, np.zeros_like(idx), idx)
        for i, j in zip(idx, js):
            perm[i], perm[j] = perm[j], perm[i]
    table = np.full((B, shape.max_pages), -1, dtype=np.int32)
    owned = np.zeros((num_pages, ps), dtype=bool)
    nxt = 0
    for b in range(B):
        for j in range(int(pages[b])):
            pg = int(perm[nxt])
            nxt += 1
            table[b, j] = pg
            owned[pg, :min(ps, int(lens[b]) - j * ps)] = True
    q = normal_tensor(seed_for(config_id, layer, "Q"), (B, shape.Hq, shape.Nq, shape.d), shape.dtype)
    pool = (num_pages, shape.Hkv, ps, shape.d)
    k = normal_tensor(seed_for(config_id, layer, "K"), pool, shape.dtype)
    v = normal_tensor(seed_for(config_id, layer, "V"), pool, shape.dtype)
    if poison:
        free = torch.from_numpy(~owned)[:, None, :, None].expand(pool)
        k = k.masked_fill(free, float("nan"))
        v = v.masked_fill(free, float("nan"))
    return q, k, v, torch.from_numpy(table), torch.from_numpy(lens.astype(np.int32))


def quantize_int8(x: torch.Tensor):
    """Symmetric per-tensor INT8 codes of x: scale = max|x| / 127 (fp32),
    codes = round-half-even(x / scale) as int8.  Returns (codes, scale)."""
    xf = x.to(torch.float32)
    amax = float(xf.abs().max())
    scale = amax / 127.0 if amax > 0 else 1.0
    scale = float(np.float32(scale))
    codes = torch.round(xf / scale).clamp_(-127, 127).to(torch.int8)
    return codes, scale


def sha256_of(t: torch.Tensor) -> str:
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return hashlib.sha256(t.numpy().tobytes()).hexdigest()


# ---------------------------------------------------------------- workloads
# The synthetic workloads (shapes, dtypes, masks, seeds).  config_id numbers
# them in a fixed order and feeds the seed rule above.
def workload_calls(name: str):
    """List of ``(AttnShape, config_id, layer)`` for a named workload."""
    if name == "mha_n64":  # smallest instance: B=1, H=2, N=64, d=64, fp16
        return [(AttnShape(1, 2, 2, 64, 64, 64, "fp16", c, 0, 0.125), 0, int(c)) for c in (False, True)]
    if name == "mha_b2h4":  # B=2, H=4, d=64, fp16, N in {256, 1024, 4096} x causal
        out = []
        for li, n in enumerate((256, 1024, 4096)):
            for c in (True, False):
                out.append((AttnShape(2, 4, 4, n, n, 64, "fp16", c, 0, None), 1, 2 * li + int(c)))
        return out
    if name == "gpt_stack":  # 12 layers of B=8, H=12, N=2048, d=64, bf16, causal, scale 1/8
        return [(AttnShape(8, 12, 12, 2048, 2048, 64, "bf16", True, 0, 0.125), 2, layer) for layer in range(12)]
    if name == "gqa_mqa":  # B=4, Hq=32, Hkv in {8, 1}, N=8192, d=128, bf16, causal; + window 4096
        return [(AttnShape(4, 32, 8, 8192, 8192, 128, "bf16", True, 0, None), 3, 0),
                (AttnShape(4, 32, 1, 8192, 8192, 128, "bf16", True, 0, None), 3, 1),
                (AttnShape(4, 32, 8, 8192, 8192, 128, "bf16", True, 4096, None), 3, 2)]
    if name == "long_prefill":  # B=1, Hq=32, Hkv=8, N=32768, d=128, bf16, keys x3, causal
        return [(AttnShape(1, 32, 8, 32768, 32768, 128, "bf16", True, 0, None, key_scale=3.0), 4, 0)]
    if name == "mqa_decode":  # one decode step: B=4, Hq=32, Hkv in {1, 8}, Nq=1, Nk=8192, d=128, bf16
        return [(AttnShape(4, 32, 1, 1, 8192, 128, "bf16", True, 0, None), 5, 0),
                (AttnShape(4, 32, 8, 1, 8192, 128, "bf16", True, 0, None), 5, 1)]
    if name == "mha_n64_bw":  # bandwidth-sized sibling of mha_n64: B=512, H=32, N=64, d=64, fp16
        return [(AttnShape(512, 32, 32, 64, 64, 64, "fp16", c, 0, 0.125), 6, int(c)) for c in (False, True)]
    if name == "mqa_decode_int8":  # mqa_decode's step on an INT8 K/V cache (per-tensor scales)
        return [(AttnShape(4, 32, 1, 1, 8192, 128, "bf16", True, 0, None, kv_int8=True), 8, 0),
                (AttnShape(4, 32, 8, 1, 8192, 128, "bf16", True, 0, None, kv_int8=True), 8, 1)]
    if name == "bwd_gpt_layer":  # the backward of a gpt_stack layer (B=8, H=12, N=2048, d=64, bf16, causal)
        return [(AttnShape(8, 12, 12, 2048, 2048, 64, "bf16", True, 0, 0.125, backward=True), 9, 0)]
    if name == "bwd_gqa":  # the backward of gqa_mqa's first call (B=4, Hq=32, Hkv=8, N=8192, d=128, bf16, causal)
        return [(AttnShape(4, 32, 8, 8192, 8192, 128, "bf16", True, 0, None, backward=True), 10, 0)]
    if name == "mla_decode":
        # one decode step of latent attention at the latent-attention section's
        # DeepSeek-V2 sizes (n_h = 128 heads, d_c = 512, scale 1/sqrt(d_h),
        # d_h = 128) on the motivation page's batch of 32 requests x 8192
        # tokens; then the same step with 4 queries per head (speculative decode)
        return [(AttnShape(32, 128, 1, 1, 8192, 512, "bf16", True, 0, 1.0 / math.sqrt(128), mla=True), 11, 0),
                (AttnShape(8, 128, 1, 4, 8192, 512, "bf16", True, 0, 1.0 / math.sqrt(128), mla=True), 11, 1)]
    if name == "paged_prefill":
        # a chunked prefill on a paged cache of 16-token pages: 2048 new query
        # rows per request against its cache of a drawn length 2048..8192
        # (the new rows are its last ones), GQA 32/8, d=128, bf16
        return [(PagedShape(4, 32, 8, 2048, 8192, 128, 16, "bf16", True, 0, None, None, 2048), 12, 0)]
    if name == "paged_decode":
        # one decode step on a paged cache of 16-token pages, bf16, d=128, GQA 32/8:
        # the mqa_decode Hkv=8 call with every request at 8192 tokens (same
        # bytes as the flat call), then a batch of 32 requests of drawn
        # lengths 512..8192 (the motivation page's batch-32, 8192-token cache)
        return [(PagedShape(4, 32, 8, 1, 8192, 128, 16, "bf16", True, 0, None, (8192,) * 4), 7, 0),
                (PagedShape(32, 32, 8, 1, 8192, 128, 16, "bf16", True, 0, None, None, 512), 7, 1)]
    raise KeyError(name)


WORKLOAD_NAMES = ["mha_n64", "mha_b2h4", "gpt_stack", "gqa_mqa", "long_prefill", "mqa_decode", "mha_n64_bw",
                  "paged_decode", "mqa_decode_int8", "bwd_gpt_layer", "bwd_gqa", "mla_decode", "paged_prefill"]
