"""The C-ABI library builds, loads and exports every symbol include/attn.h
declares; host-side validation answers without touching a GPU."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def attn():
    import tiled_attention_forward_fwd_gb300 as m

    m.lib()
    return m


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_symbols_exported(attn):
    names = declared_functions()
    assert len(names) >= 9, names
    L = attn.lib()
    for n in names:
        assert hasattr(L, n), f"libattn.so does not export {n}"
    assert sorted(attn.EXPORTED) == names


def test_abi_version_and_strings(attn):
    assert attn.attn_abi_version() == 1
    for code, text in [(0, "ok"), (1, "invalid argument"), (3, "CUDA error"), (4, "kernel wait timed out")]:
        assert attn.attn_status_string(code) == text
    assert attn.attn_status_string(99) == "unknown status"


FAKE = 1 << 20  # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("args,expect", [
    (dict(B=1, Hq=3, Hkv=2), 1),             # Hq % Hkv
    (dict(B=0), 1),                            # empty batch
    (dict(N=0), 1),
    (dict(d=96), 2),                           # unsupported head dim
    (dict(window=-1), 1),
    (dict(window=16, causal=0), 1),            # window needs causal
    (dict(sm_scale=0.0), 1),
    (dict(sm_scale=float("inf")), 1),
    (dict(sm_scale=float("nan")), 1),
    (dict(dtype=7), 1),
])
def test_host_validation(attn, args, expect):
    a = dict(B=1, Hq=2, Hkv=2, N=64, d=64, causal=1, window=0, sm_scale=0.125, dtype=0)
    a.update(args)
    st = attn.attn_fwd(FAKE, FAKE, FAKE, FAKE, None, a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["causal"],
                       a["window"], a["sm_scale"], a["dtype"], None)
    assert st == expect


def test_null_and_misaligned_pointers(attn):
    assert attn.attn_fwd(None, FAKE, FAKE, FAKE, None, 1, 2, 2, 64, 64, 0, 0, 0.1, 0, None) == 1
    assert attn.attn_fwd(FAKE + 8, FAKE, FAKE, FAKE, None, 1, 2, 2, 64, 64, 0, 0, 0.1, 0, None) == 1
    assert attn.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE + 2, 1, 2, 2, 64, 64, 0, 0, 0.1, 0, None) == 1
    # causal with more queries than keys
    assert attn.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 65, 64, 64, 1, 0, 0.1, 0, None, 0, None) == 1
    # host entry: null host buffer, unaligned staging buffer, staging too small
    assert attn.attn_fwd_host(None, FAKE, FAKE, FAKE, None, 1, 2, 2, 64, 64, 64, 0, 0, 0.1, 0, FAKE, 1 << 30,
                              None) == 1
    assert attn.attn_fwd_host(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 64, 64, 64, 0, 0, 0.1, 0, FAKE + 16, 1 << 30,
                              None) == 1
    assert attn.attn_fwd_host(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 64, 64, 64, 0, 0, 0.1, 0, FAKE, 100,
                              None) == 1


def test_sizes(attn):
    # staging = Q + K + V + O (+ LSE), each rounded up to 256 bytes
    q = 1 * 2 * 64 * 64 * 2
    assert attn.attn_fwd_host_staging_bytes(1, 2, 2, 64, 64, 64, 0) == 4 * q
    assert attn.attn_fwd_host_staging_bytes(1, 2, 2, 64, 64, 64, 1) == 4 * q + 512
    assert attn.attn_fwd_host_staging_bytes(0, 2, 2, 64, 64, 64, 1) == 0
    assert attn.attn_fwd_workspace_bytes(1, 2, 3, 1, 64, 64) == 0  # Hq % Hkv


@pytest.mark.parametrize("change", [
    dict(table=None),                  # no page table
    dict(lens=FAKE + 2),               # misaligned lengths
    dict(page_size=12),                # not a power of two
    dict(page_size=4),                 # below 8
    dict(page_size=512),               # above 256
    dict(num_pages=0),
    dict(max_pages=3),                 # 3 pages of 16 cannot cover 64 tokens
    dict(num_pages=1 << 30, Hkv=2),    # pool slabs past 32-bit copy coordinates
    dict(window=8, causal=0),          # window needs causal
    dict(Nq=65),                       # causal with more queries than keys
    dict(Hq=3),                        # Hq % Hkv
])
def test_paged_host_validation(attn, change):
    """attn_fwd_paged rejects bad arguments on the host, before touching the
    device (the pointers are never dereferenced)."""
    a = dict(table=FAKE, lens=FAKE, B=2, Hq=8, Hkv=2, Nq=1, max_len=64, d=128, page_size=16, num_pages=8,
             max_pages=4, causal=1, window=0)
    a.update(change)
    st = attn.attn_fwd_paged(FAKE, FAKE, FAKE, a["table"], a["lens"], FAKE, None, a["B"], a["Hq"], a["Hkv"], a["Nq"],
                             a["max_len"], a["d"], a["page_size"], a["num_pages"], a["max_pages"], a["causal"],
                             a["window"], 0.1, 1, FAKE, 1 << 20, None)
    assert st == attn.ATTN_ERR_INVALID_ARG


def test_paged_status_string(attn):
    assert "page index" in attn.attn_status_string(attn.ATTN_ERR_DEVICE_ARG)
    assert attn.attn_fwd_paged_workspace_bytes(1, 3, 2, 1, 64, 128) == 0  # Hq % Hkv
    assert attn.attn_fwd_paged_workspace_bytes(1, 2, 2, 1, 64, 96) == 0   # head dim


def test_maximum_sizes_rejected(attn):
    """Work items are counted in 32 bits: a call with more than 2^31 - 1
    query tiles (B * Hq * ceil(Nq / 128)) is rejected on the host, before any
    launch (the pointers are never used, on any machine)."""
    too_many = attn.attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 65536, 256, 256, 1 << 20, 64, 1, 0, 0.125, 0, None)
    assert too_many == attn.ATTN_ERR_INVALID_ARG
    B, H, N = 16384, 1024, 16384  # 16384 * 1024 * 128 tiles = 2^31, one past the limit
    assert attn.attn_fwd(FAKE, FAKE, FAKE, FAKE, None, B, H, H, N, 64, 0, 0, 0.125, 0, None) == attn.ATTN_ERR_INVALID_ARG
    # the schedule query refuses item lists past 32 bits as well
    assert attn.attn_fwd_prefill_visits(65536, 256, 256, 1 << 20, 1 << 20, 64, 1, 0, 0, 152) is None


def test_size_queries_do_not_overflow(attn):
    """Byte counts are 64-bit: a 2^31-element tensor's staging size is exact."""
    B, H, N, d = 4, 32, 131072, 128  # Q is 2^31 elements
    q_bytes = B * H * N * d * 2
    got = attn.attn_fwd_host_staging_bytes(B, H, H, N, N, d, 1)
    lse = B * H * N * 4
    assert got >= 4 * q_bytes + lse and got < 4 * q_bytes + lse + 5 * 256 + (1 << 30)
