"""Algorithmic work of the attention hot path: effective FLOPs and decode bytes.

Effective prefill FLOPs count only the (query, key) pairs the mask lets through:
4 d per pair and query head (2 d for Q.K, 2 d for P.V), the way the pages count decode
compute ("PLaMo 3アーキテクチャ徹底解析" §2.3: dot products and weighted sums, 2 FLOP per
multiply-add, i.e. 4 B H_q d A).  Masked pairs inside partially masked tiles are work the
kernel does but does not get credit for.

Decode bytes follow the same section: every cached K and V is read once per (sequence,
KV head), shared by the G query heads of its group: 4 Hkv d bytes per token and layer
in bf16 (2 for K and V, 2 bytes each).
"""
from __future__ import annotations

from typing import Iterable


def unmasked_pairs(T: int, S: int, window: int) -> int:
    """Number of visible (query, key) pairs for one (batch, head): queries at positions
    S-T..S-1, each sees min(position + 1, window) keys (window <= 0: position + 1)."""
    lo, hi = S - T + 1, S          # position + 1 over the query rows
    if window <= 0 or window >= hi:
        return (lo + hi) * (hi - lo + 1) // 2
    total = 0
    top = min(hi, window - 1)
    if top >= lo:
        total += (lo + top) * (top - lo + 1) // 2
    n_full = hi - max(lo, window) + 1
    if n_full > 0:
        total += n_full * window
    return total


def prefill_flops(B: int, Hq: int, T: int, S: int, d: int, window: int) -> int:
    return 4 * d * B * Hq * unmasked_pairs(T, S, window)


def decode_kv_bytes(retained: Iterable[int], Hkv: int, d: int, elem_bytes: int = 2,
                    kv_shared: bool = False) -> int:
    """K and V bytes one decode step must read: 2 Hkv d elem_bytes per retained token, or
    half that when K and V share one cached row (Gemma 4 global layers)."""
    rows = 1 if kv_shared else 2
    return sum(rows * int(r) * Hkv * d * elem_bytes for r in retained)


def kv_bytes_per_token(L: int, Hkv: int, d: int, N: int, W: int, elem_bytes: int = 2) -> int:
    """Decode K/V reads per generated token over a whole hybrid model (§2.3): global
    layers N_g = L/8 read N tokens, local layers N_l = 7L/8 read min(N, W); the same
    formula gives the cache capacity of §5.2."""
    n_g, n_l = L // 8, 7 * L // 8
    return 2 * elem_bytes * Hkv * d * (n_g * N + n_l * min(N, W))


def kv_capacity_bytes(layers, N: int, elem_bytes: int = 2) -> int:
    """Cache bytes for a list of (n_layers, Hkv, d, window or 0) groups at length N."""
    total = 0
    for n, hkv, d, w in layers:
        tokens = N if w <= 0 else min(N, w)
        total += 2 * elem_bytes * n * hkv * d * tokens
    return total


def _short_items(T: int, S: int, window: int) -> bool:
    """Whether the 128-row query blocks average fewer than 48 key tiles (windowed layers,
    short sequences): the library's launchers then pick their persistent kernels."""
    n_mb = -(-T // 128)
    tiles = 0
    for mb in range(n_mb):
        q_lo = S - T + mb * 128
        q_hi = min(q_lo + 127, S - 1)
        kt0 = max(0, q_lo - window + 1) // 128 if window > 0 else 0
        tiles += q_hi // 128 - kt0 + 1
    return tiles < 48 * n_mb


def prefill_d128_kernel(T: int, S: int, window: int) -> str:
    """Which d = 128 prefill kernel the library launches for these positions: the
    one-CTA-per-item kernel when the 128-row query blocks average at least 48 key tiles
    (long causal sweeps), the persistent kernel otherwise.  Mirrors the rule in the
    library's launcher; used to label measurements."""
    return "prefill_persistent_kernel" if _short_items(T, S, window) else "prefill_kernel"


def prefill_kernel_name(d: int, T: int, S: int, window: int) -> str:
    """The prefill kernel the library launches for head dim d at these positions."""
    if d == 128:
        return prefill_d128_kernel(T, S, window)
    if d == 512:
        return "prefill_pair_kernel"
    return f"prefill_wide_kernel<{d}>"
