"""Tiled (FlashAttention) forward pass for NVIDIA GB300 (sm_103a).

Thin ctypes binding over ``libattn.so`` (C ABI in ``include/attn.h``).  The
functions below keep the C names and only marshal arguments; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library cannot be built or loaded, importing this package raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import math
import threading

from . import _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_SCRATCH_LIMIT = 5
ATTN_ERR_DEVICE_ARG = 6

ATTN_DTYPE_FP16 = 0
ATTN_DTYPE_BF16 = 1

ATTN_PATH_PREFILL = 0
ATTN_PATH_SPLIT_KV = 1
ATTN_PATH_SHORT = 2
ATTN_PATH_PREFILL_SPLIT = 3
ATTN_PATH_SPLIT_KV_FUSED = 4

EXPORTED = ["attn_fwd", "attn_fwd_ex", "attn_fwd_workspace_bytes", "attn_fwd_host", "attn_fwd_host_staging_bytes",
            "attn_device_status", "attn_set_wait_timeout_ns", "attn_status_string", "attn_abi_version",
            "attn_fwd_decode_noalloc", "attn_fwd_path", "attn_fwd_prefill_visits", "attn_fwd_paged",
            "attn_fwd_paged_workspace_bytes", "attn_fwd_paged_path",
            "attn_fwd_decode_plan", "attn_set_test_stall", "attn_fwd_kv_int8", "attn_bwd", "attn_bwd_workspace_bytes",
            "attn_fwd_mla", "attn_fwd_mla_workspace_bytes", "attn_empty_launch", "attn_fwd_kv_int8_workspace_bytes",
            "attn_bwd_cta_order"]

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {attn_status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """Load (building first if needed) libattn.so.  Raises if unavailable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        fp = ctypes.POINTER(ctypes.c_float)
        L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp]
        L.attn_fwd.restype = ci
        L.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp, sz, vp]
        L.attn_fwd_ex.restype = ci
        L.attn_fwd_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
        L.attn_fwd_workspace_bytes.restype = sz
        L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp, sz, vp]
        L.attn_fwd_host.restype = ci
        L.attn_fwd_host_staging_bytes.argtypes = [ci, ci, ci, ci, ci, ci, ci]
        L.attn_fwd_host_staging_bytes.restype = sz
        L.attn_device_status.argtypes = [vp]
        L.attn_device_status.restype = ci
        L.attn_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        L.attn_set_wait_timeout_ns.restype = None
        L.attn_set_test_stall.argtypes = [ci]
        L.attn_set_test_stall.restype = None
        L.attn_fwd_kv_int8.argtypes = [vp, vp, vp, cf, cf, vp, vp] + [ci] * 8 + [cf, ci, vp, sz, vp]
        L.attn_fwd_kv_int8.restype = ci
        L.attn_fwd_kv_int8_workspace_bytes.argtypes = [ci] * 6
        L.attn_fwd_kv_int8_workspace_bytes.restype = sz
        L.attn_bwd.argtypes = [vp] * 9 + [ci] * 8 + [cf, ci, vp, sz, vp]
        L.attn_bwd.restype = ci
        L.attn_bwd_workspace_bytes.argtypes = [ci] * 4
        L.attn_bwd_workspace_bytes.restype = sz
        L.attn_bwd_cta_order.argtypes = [ci, ci, ci, ci, ctypes.POINTER(ci), ci]
        L.attn_bwd_cta_order.restype = ci
        L.attn_fwd_mla.argtypes = [vp, vp, vp, vp] + [ci] * 7 + [cf, ci, vp, sz, vp]
        L.attn_fwd_mla.restype = ci
        L.attn_fwd_mla_workspace_bytes.argtypes = [ci] * 5
        L.attn_fwd_mla_workspace_bytes.restype = sz
        L.attn_empty_launch.argtypes = [ci, ci, sz, vp]
        L.attn_empty_launch.restype = ci
        L.attn_status_string.argtypes = [ci]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_abi_version.argtypes = []
        L.attn_abi_version.restype = ci
        L.attn_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf, ci, vp]
        L.attn_fwd_decode_noalloc.restype = ci
        L.attn_fwd_path.argtypes = [ci, ci, ci, ci, ci, ci, ci]
        L.attn_fwd_path.restype = ci
        L.attn_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp] + [ci] * 11 + [cf, ci, vp, sz, vp]
        L.attn_fwd_paged.restype = ci
        L.attn_fwd_paged_workspace_bytes.argtypes = [ci] * 6
        L.attn_fwd_paged_workspace_bytes.restype = sz
        L.attn_fwd_paged_path.argtypes = [ci] * 6
        L.attn_fwd_paged_path.restype = ci
        L.attn_fwd_decode_plan.argtypes = [ci] * 9 + [ctypes.POINTER(ctypes.c_longlong)]
        L.attn_fwd_decode_plan.restype = ci
        ip = ctypes.POINTER(ctypes.c_int)
        L.attn_fwd_prefill_visits.argtypes = [ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, ip, ip, ci]
        L.attn_fwd_prefill_visits.restype = ci
        del fp
        _lib = L
        return _lib


# ------------------------------------------------------------------ raw C names
def attn_fwd(Q, K, V, O, LSE, B, Hq, Hkv, N, d, causal, window, sm_scale, dtype, stream) -> int:
    return lib().attn_fwd(Q, K, V, O, LSE, B, Hq, Hkv, N, d, int(causal), int(window), float(sm_scale), int(dtype),
                          stream)


def attn_fwd_ex(Q, K, V, O, LSE, B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype, workspace,
                workspace_bytes, stream) -> int:
    return lib().attn_fwd_ex(Q, K, V, O, LSE, B, Hq, Hkv, Nq, Nk, d, int(causal), int(window), float(sm_scale),
                             int(dtype), workspace, int(workspace_bytes), stream)


def attn_fwd_workspace_bytes(B, Hq, Hkv, Nq, Nk, d) -> int:
    return int(lib().attn_fwd_workspace_bytes(B, Hq, Hkv, Nq, Nk, d))


def attn_fwd_path(B, Hq, Hkv, Nq, Nk, d, with_workspace) -> int:
    return int(lib().attn_fwd_path(B, Hq, Hkv, Nq, Nk, d, 1 if with_workspace else 0))


def attn_fwd_decode_plan(B, Hq, Hkv, Nq, Nk, d, paged, sms, ctas_per_sm):
    """The split-KV plan without device work: dict(nchunks, chunk_keys,
    fused, flag_off, bytes), or None when the shape takes no split-KV path.
    ``paged``: False / 0 flat cache, True / 1 paged cache, 2 int8 cache."""
    info = (ctypes.c_longlong * 5)()
    if lib().attn_fwd_decode_plan(B, Hq, Hkv, Nq, Nk, d, int(paged), sms, ctas_per_sm, info) != 0:
        return None
    return dict(zip(("nchunks", "chunk_keys", "fused", "flag_off", "bytes"), (int(x) for x in info)))


def attn_fwd_prefill_visits(B, Hq, Hkv, Nq, Nk, d, causal, window, with_workspace, sms):
    """The prefill schedule without device work: (info, visits) with info =
    (grid, schedule, item shape, items) and visits an (n, 6) int32 array of
    (cta, item, tile slot, b * Hq + h, first query row, K/V tile) in launch
    order; None when the sizes take no prefill path."""
    import numpy as np

    info = (ctypes.c_int * 4)()
    args = (B, Hq, Hkv, Nq, Nk, d, int(causal), int(window), 1 if with_workspace else 0, sms)
    n = lib().attn_fwd_prefill_visits(*args, info, None, 0)
    if n < 0:
        return None
    visits = np.zeros((max(n, 1), 6), dtype=np.int32)
    got = lib().attn_fwd_prefill_visits(*args, info, visits.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n)
    if got != n:
        raise RuntimeError("attn_fwd_prefill_visits: visit count changed between calls")
    return tuple(info), visits[:n]


def attn_fwd_paged(Q, K_pages, V_pages, block_table, seq_lens, O, LSE, B, Hq, Hkv, Nq, max_seq_len, d, page_size,
                   num_pages, max_pages_per_seq, causal, window, sm_scale, dtype, workspace, workspace_bytes,
                   stream) -> int:
    return lib().attn_fwd_paged(Q, K_pages, V_pages, block_table, seq_lens, O, LSE, B, Hq, Hkv, Nq, max_seq_len, d,
                                page_size, num_pages, max_pages_per_seq, int(causal), int(window), float(sm_scale),
                                int(dtype), workspace, int(workspace_bytes), stream)


def attn_fwd_kv_int8(Q, K_codes, V_codes, k_scale, v_scale, O, LSE, B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale,
                     dtype, workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd_kv_int8(Q, K_codes, V_codes, float(k_scale), float(v_scale), O, LSE, B, Hq, Hkv, Nq, Nk, d,
                                  int(causal), int(window), float(sm_scale), int(dtype), workspace,
                                  int(workspace_bytes), stream)


def attn_fwd_kv_int8_workspace_bytes(B, Hq, Hkv, Nq, Nk, d) -> int:
    return int(lib().attn_fwd_kv_int8_workspace_bytes(B, Hq, Hkv, Nq, Nk, d))


def attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype, workspace,
             workspace_bytes, stream) -> int:
    return lib().attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, Nq, Nk, d, int(causal), int(window),
                          float(sm_scale), int(dtype), workspace, int(workspace_bytes), stream)


def attn_bwd_workspace_bytes(B, Hq, Nq, d) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, Hq, Nq, d))


def attn_bwd_cta_order(B, Hkv, Nk, sms):
    """The backward kernel's CTA order: an int array (CTAs, 2) of (K/V group,
    key tile) in launch order, or None for bad sizes."""
    import numpy as np

    n = int(lib().attn_bwd_cta_order(B, Hkv, Nk, sms, None, 0))
    if n < 0:
        return None
    out = np.zeros((n, 2), dtype=np.int32)
    got = int(lib().attn_bwd_cta_order(B, Hkv, Nk, sms, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n))
    assert got == n
    return out


def attn_fwd_mla(Q_lat, C_lat, O_lat, LSE, B, n_h, Nq, Nk, d_c, causal, window, sm_scale, dtype, workspace,
                 workspace_bytes, stream) -> int:
    return lib().attn_fwd_mla(Q_lat, C_lat, O_lat, LSE, B, n_h, Nq, Nk, d_c, int(causal), int(window),
                              float(sm_scale), int(dtype), workspace, int(workspace_bytes), stream)


def attn_empty_launch(grid, threads, smem_bytes, stream) -> int:
    return int(lib().attn_empty_launch(int(grid), int(threads), int(smem_bytes), stream))


def attn_fwd_mla_workspace_bytes(B, n_h, Nq, Nk, d_c) -> int:
    return int(lib().attn_fwd_mla_workspace_bytes(B, n_h, Nq, Nk, d_c))


def attn_fwd_paged_workspace_bytes(B, Hq, Hkv, Nq, max_seq_len, d) -> int:
    return int(lib().attn_fwd_paged_workspace_bytes(B, Hq, Hkv, Nq, max_seq_len, d))


def attn_fwd_paged_path(B, Hq, Hkv, Nq, max_seq_len, d) -> int:
    return int(lib().attn_fwd_paged_path(B, Hq, Hkv, Nq, max_seq_len, d))


def attn_fwd_host(Qh, Kh, Vh, Oh, LSEh, B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype, dev_buf,
                  dev_buf_bytes, stream) -> int:
    return lib().attn_fwd_host(Qh, Kh, Vh, Oh, LSEh, B, Hq, Hkv, Nq, Nk, d, int(causal), int(window),
                               float(sm_scale), int(dtype), dev_buf, int(dev_buf_bytes), stream)


def attn_fwd_host_staging_bytes(B, Hq, Hkv, Nq, Nk, d, with_lse) -> int:
    return int(lib().attn_fwd_host_staging_bytes(B, Hq, Hkv, Nq, Nk, d, int(bool(with_lse))))


def attn_device_status(stream) -> int:
    return int(lib().attn_device_status(stream))


def attn_set_wait_timeout_ns(ns: int) -> None:
    lib().attn_set_wait_timeout_ns(int(ns))


def attn_set_test_stall(tiles: int) -> None:
    lib().attn_set_test_stall(int(tiles))


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_abi_version() -> int:
    return int(lib().attn_abi_version())


def attn_fwd_decode_noalloc(Q, K, V, O, LSE, B, Hq, Hkv, Nq, Nk, d, causal, window, sm_scale, dtype,
                            stream) -> int:
    """Split-KV decode whose scratch is a fixed block inside the library (for
    callers that cannot provide device memory); see include/attn.h."""
    return lib().attn_fwd_decode_noalloc(Q, K, V, O, LSE, B, Hq, Hkv, Nq, Nk, d, int(causal), int(window),
                                         float(sm_scale), int(dtype), stream)


# ------------------------------------------------------------------ torch-facing
def _torch():
    import torch

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return ATTN_DTYPE_FP16
    if t.dtype == torch.bfloat16:
        return ATTN_DTYPE_BF16
    raise TypeError(f"attention inputs must be float16 or bfloat16, got {t.dtype}")


def _stream_handle(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def flash_attn_forward(q, k, v, causal: bool = False, window: int = 0, sm_scale: float | None = None,
                       return_lse: bool = True, out=None, lse=None, workspace=None):
    """O = softmax(sm_scale * q k^T + mask) v on CUDA tensors.

    q: (B, Hq, Nq, d); k, v: (B, Hkv, Nk, d); fp16 or bf16, same dtype and
    device.  ``sm_scale`` defaults to 1/sqrt(d).  Returns ``(O, LSE)`` (LSE is
    fp32 (B, Hq, Nq), or None when ``return_lse`` is False).  ``workspace`` (a
    CUDA byte tensor of ``attn_fwd_workspace_bytes`` bytes) enables the
    split-KV path for small query counts.  Runs on the current stream."""
    torch = _torch()
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("flash_attn_forward needs CUDA tensors (no CPU path)")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be (B,Hq,Nq,d) and k, v (B,Hkv,Nk,d)")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k, v batch / head dim do not match q")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                     lse.data_ptr() if return_lse else None, B, Hq, Hkv, Nq, Nk, d, causal, window, scale,
                     _dtype_code(q), ws_ptr, ws_bytes, _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_ex")
    return out, (lse if return_lse else None)


def flash_attn_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len: int, causal: bool = True,
                     window: int = 0, sm_scale: float | None = None, return_lse: bool = True, out=None, lse=None,
                     workspace=None):
    """Attention over a paged K/V cache on CUDA tensors (see attn_fwd_paged
    in include/attn.h).

    q: (B, Hq, Nq, d); k_pages, v_pages: (num_pages, Hkv, page_size, d), same
    dtype (fp16 or bf16); block_table: (B, max_pages) int32; seq_lens: (B,)
    int32, all on q's device.  Row i of request b sits at position
    seq_lens[b] - Nq + i.  ``workspace`` (a CUDA byte tensor of at least
    ``attn_fwd_paged_workspace_bytes`` bytes) is allocated when not given.
    Returns ``(O, LSE)``.  Runs on the current stream."""
    torch = _torch()
    ts = (q, k_pages, v_pages, block_table, seq_lens)
    if not all(t.is_cuda for t in ts):
        raise ValueError("flash_attn_paged needs CUDA tensors (no CPU path)")
    if not (q.dtype == k_pages.dtype == v_pages.dtype):
        raise TypeError("q and the page pools must share a dtype")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if q.dim() != 4 or k_pages.dim() != 4 or k_pages.shape != v_pages.shape or block_table.dim() != 2:
        raise ValueError("q must be (B,Hq,Nq,d), pools (num_pages,Hkv,page_size,d), block_table (B,max_pages)")
    q, k_pages, v_pages = q.contiguous(), k_pages.contiguous(), v_pages.contiguous()
    block_table, seq_lens = block_table.contiguous(), seq_lens.contiguous()
    B, Hq, Nq, d = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if k_pages.shape[3] != d or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("pools, table or lengths do not match q")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    if workspace is None:
        need = attn_fwd_paged_workspace_bytes(B, Hq, Hkv, Nq, max_seq_len, d)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = attn_fwd_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(),
                        seq_lens.data_ptr(), out.data_ptr(), lse.data_ptr() if return_lse else None, B, Hq, Hkv, Nq,
                        max_seq_len, d, page_size, num_pages, block_table.shape[1], causal, window, scale,
                        _dtype_code(q), workspace.data_ptr(), workspace.numel(), _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_paged")
    return out, (lse if return_lse else None)


def flash_attn_kv_int8(q, k_codes, v_codes, k_scale: float, v_scale: float, causal: bool = True, window: int = 0,
                      sm_scale: float | None = None, return_lse: bool = True, out=None, lse=None, workspace=None):
    """Decode over an INT8 K/V cache (see attn_fwd_kv_int8 in include/attn.h):
    K = k_scale * k_codes, V = v_scale * v_codes.  q: (B, Hq, Nq, d) fp16 or
    bf16; k_codes, v_codes: (B, Hkv, Nk, d) int8, on q's device.
    ``workspace`` (a CUDA byte tensor of at least
    ``attn_fwd_kv_int8_workspace_bytes`` bytes) is allocated when not given.  Returns ``(O, LSE)``.  Runs on the
    current stream."""
    torch = _torch()
    if not (q.is_cuda and k_codes.is_cuda and v_codes.is_cuda):
        raise ValueError("flash_attn_kv_int8 needs CUDA tensors (no CPU path)")
    if k_codes.dtype != torch.int8 or v_codes.dtype != torch.int8:
        raise TypeError("k_codes and v_codes must be int8")
    if q.dim() != 4 or k_codes.dim() != 4 or k_codes.shape != v_codes.shape:
        raise ValueError("q must be (B,Hq,Nq,d) and the codes (B,Hkv,Nk,d)")
    q, k_codes, v_codes = q.contiguous(), k_codes.contiguous(), v_codes.contiguous()
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k_codes.shape[1], k_codes.shape[2]
    if k_codes.shape[0] != B or k_codes.shape[3] != d:
        raise ValueError("codes batch / head dim do not match q")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    if workspace is None:
        need = attn_fwd_kv_int8_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = attn_fwd_kv_int8(q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(), k_scale, v_scale, out.data_ptr(),
                          lse.data_ptr() if return_lse else None, B, Hq, Hkv, Nq, Nk, d, causal, window, scale,
                          _dtype_code(q), workspace.data_ptr(), workspace.numel(), _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_kv_int8")
    return out, (lse if return_lse else None)


def flash_attn_mla(q_lat, c_lat, causal: bool = True, window: int = 0, sm_scale: float | None = None,
                   return_lse: bool = True, out=None, lse=None, workspace=None):
    """Attention over a latent cache with absorbed queries (see attn_fwd_mla
    in include/attn.h).  q_lat: (B, n_h, Nq, d_c) fp16 or bf16, the absorbed
    queries; c_lat: (B, Nk, d_c), same dtype and device; d_c = 512.
    ``sm_scale`` defaults to 1/sqrt(d_c); a model passes its own (the head
    dimension's).  Returns ``(O_lat, LSE)``, O_lat (B, n_h, Nq, d_c).  Runs on
    the current stream."""
    torch = _torch()
    if not (q_lat.is_cuda and c_lat.is_cuda):
        raise ValueError("flash_attn_mla needs CUDA tensors (no CPU path)")
    if q_lat.dtype != c_lat.dtype:
        raise TypeError("q_lat and c_lat must share a dtype")
    if q_lat.dim() != 4 or c_lat.dim() != 3:
        raise ValueError("q_lat must be (B,n_h,Nq,d_c) and c_lat (B,Nk,d_c)")
    q_lat, c_lat = q_lat.contiguous(), c_lat.contiguous()
    B, n_h, Nq, d_c = q_lat.shape
    Nk = c_lat.shape[1]
    if c_lat.shape[0] != B or c_lat.shape[2] != d_c:
        raise ValueError("c_lat batch / latent width do not match q_lat")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(d_c)
    if out is None:
        out = torch.empty_like(q_lat)
    if return_lse and lse is None:
        lse = torch.empty((B, n_h, Nq), device=q_lat.device, dtype=torch.float32)
    if workspace is None:
        need = attn_fwd_mla_workspace_bytes(B, n_h, Nq, Nk, d_c)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_lat.device)
    st = attn_fwd_mla(q_lat.data_ptr(), c_lat.data_ptr(), out.data_ptr(), lse.data_ptr() if return_lse else None,
                      B, n_h, Nq, Nk, d_c, causal, window, scale, _dtype_code(q_lat), workspace.data_ptr(),
                      workspace.numel(), _stream_handle(q_lat.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_mla")
    return out, (lse if return_lse else None)


def flash_attn_backward(q, k, v, o, lse, do, causal: bool = False, window: int = 0, sm_scale: float | None = None,
                        workspace=None):
    """Gradients (dQ, dK, dV) of O = softmax(sm_scale * q k^T + mask) v for an
    upstream gradient ``do`` (see attn_bwd in include/attn.h).  ``o`` and
    ``lse`` are the forward's outputs for the same arguments.  dK and dV sum
    the query heads of each K/V head.  Runs on the current stream."""
    torch = _torch()
    ts = (q, k, v, o, do)
    if not all(t.is_cuda for t in ts) or not lse.is_cuda:
        raise ValueError("flash_attn_backward needs CUDA tensors (no CPU path)")
    if not all(t.dtype == q.dtype for t in ts) or lse.dtype != torch.float32:
        raise TypeError("q, k, v, o, do must share a dtype; lse must be float32")
    q, k, v, o, do, lse = (t.contiguous() for t in (q, k, v, o, do, lse))
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if o.shape != q.shape or do.shape != q.shape or v.shape != k.shape or lse.shape != (B, Hq, Nq):
        raise ValueError("inconsistent shapes")
    scale = float(sm_scale) if sm_scale is not None else 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(max(attn_bwd_workspace_bytes(B, Hq, Nq, d), 16), dtype=torch.uint8, device=q.device)
    st = attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Nq, Nk, d, causal, window, scale,
                  _dtype_code(q), workspace.data_ptr(), workspace.numel(), _stream_handle(q.device))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def device_status(device=None) -> int:
    """Synchronise the current stream and read/clear the kernel status word."""
    return attn_device_status(_stream_handle(device))


__all__ = EXPORTED + ["flash_attn_forward", "flash_attn_paged", "flash_attn_kv_int8", "flash_attn_backward",
                      "device_status", "lib", "AttnError"]
