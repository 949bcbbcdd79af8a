"""Work and traffic accounting for throughput and roofline figures.

FLOPs: 4*d per live (query, key) pair -- two multiply-adds per element of
S = Q K^T and of P V (motivation page, "Por que la attention es
bandwidth-bound": 4 N^2 d per head).  The headline metric counts a square
causal problem as half of the full one (4*B*Hq*N^2*d / 2); every other case
(sliding window, Nq != Nk) counts the exact live pairs.

Bytes: the compulsory traffic of the method -- Q, K, V read once, O written
once, LSE written once.  The score matrix never reaches memory, so it is not
counted; re-reads of K/V tiles that hit L2 are an implementation cost, not
algorithmic work.
"""
from __future__ import annotations


def live_pairs_per_head(Nq: int, Nk: int, causal: bool, window: int) -> int:
    """Number of (query, key) pairs that survive the mask, for one (b, h)."""
    if not causal:
        return Nq * Nk
    off = Nk - Nq
    total = 0
    # rows i: position p = off + i sees keys max(0, p - window + 1) .. p (window > 0), else 0 .. p
    if window <= 0:
        # sum_{i} (off + i + 1) for off + i >= 0
        first = max(0, -off)
        n = Nq - first
        if n <= 0:
            return 0
        a = off + first + 1
        return n * a + n * (n - 1) // 2
    for i in range(Nq):
        p = off + i
        if p < 0:
            continue
        total += min(p + 1, window)
    return total


def metric_flops(B: int, Hq: int, Nq: int, Nk: int, d: int, causal: bool, window: int = 0) -> float:
    """FLOPs under the headline convention (square causal = half of full)."""
    if Nq == Nk and window <= 0:
        full = 4.0 * B * Hq * Nq * Nk * d
        return full / 2.0 if causal else full
    return 4.0 * B * Hq * d * live_pairs_per_head(Nq, Nk, causal, window)


def exact_flops(B: int, Hq: int, Nq: int, Nk: int, d: int, causal: bool, window: int = 0) -> float:
    return 4.0 * B * Hq * d * live_pairs_per_head(Nq, Nk, causal, window)


def compulsory_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, elem_bytes: int = 2,
                     with_lse: bool = True) -> int:
    b = elem_bytes * d * (2 * B * Hq * Nq + 2 * B * Hkv * Nk)
    if with_lse:
        b += 4 * B * Hq * Nq
    return b


def shape_flops(s, exact: bool = False) -> float:
    """The forward's FLOPs; for a backward call (s.backward) 2.5 times as
    many: five matrix products of the forward's size (S, dP, dV, dK, dQ)
    against its two."""
    f = exact_flops if exact else metric_flops
    fw = f(s.B, s.Hq, s.Nq, s.Nk, s.d, s.causal, s.window)
    return 2.5 * fw if getattr(s, "backward", False) else fw


def shape_bytes(s, with_lse: bool = True) -> int:
    if getattr(s, "backward", False):
        # reads Q, O, dO and K, V; writes dQ and dK, dV; reads the LSE
        b = 2 * s.d * (4 * s.B * s.Hq * s.Nq + 4 * s.B * s.Hkv * s.Nk)
        return b + (4 * s.B * s.Hq * s.Nq if with_lse else 0)
    if getattr(s, "mla", False):  # latent attention: one latent cache (B, Nk, d_c) serves as K and V
        b = 2 * s.d * (2 * s.B * s.Hq * s.Nq + s.B * s.Nk)
        return b + (4 * s.B * s.Hq * s.Nq if with_lse else 0)
    if getattr(s, "kv_int8", False):  # Q and O 16-bit, K and V one byte per element
        b = 2 * s.d * 2 * s.B * s.Hq * s.Nq + s.d * 2 * s.B * s.Hkv * s.Nk
        return b + (4 * s.B * s.Hq * s.Nq if with_lse else 0)
    return compulsory_bytes(s.B, s.Hq, s.Hkv, s.Nq, s.Nk, s.d, 2, with_lse)


def paged_flops(s, lens) -> float:
    """Exact FLOPs of a paged-cache call (ai.PagedShape s, per-request key
    counts lens): each request's live pairs at its own length."""
    return 4.0 * s.Hq * s.d * sum(live_pairs_per_head(s.Nq, int(n), s.causal, s.window) for n in lens)


def paged_bytes(s, lens, with_lse: bool = True) -> int:
    """Compulsory traffic of a paged-cache call: Q and O once, each request's
    K and V tokens once (its length, not the pool), its page-table entries
    and its length (4 bytes each), and the LSE."""
    b = 2 * s.d * (2 * s.B * s.Hq * s.Nq + 2 * s.Hkv * sum(int(n) for n in lens))
    b += 4 * sum(-(-int(n) // s.page_size) for n in lens) + 4 * s.B
    if with_lse:
        b += 4 * s.B * s.Hq * s.Nq
    return b


# Page formulas (used to pin the accounting against the pages' printed numbers).
def naive_score_traffic_bytes(N: int) -> int:
    """fp32 S written, read, written, read: 16 N^2 bytes (motivation page)."""
    return 16 * N * N


def flash_traffic_bytes_fp32(N: int, d: int, Bc: int) -> float:
    """The motivation page's estimate N*d*(3 + 2N/B_c)*4 bytes."""
    return N * d * (3 + 2 * N / Bc) * 4
