"""Helpers for the GPU tests: device buffers, RoPE tables, calls through the C-ABI binding,
and comparison against the fp64 oracle at the stated tolerance."""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import oracle as oracle_pkg
from workloads import RopeSpec

# Parity bar on bf16 outputs (fp32 accumulation) against the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if gqa.gqa_device_check() != 0:
        pytest.skip("device is not sm_103")


def orc():
    return oracle_pkg.default()


def rope_table(d: int, rope: RopeSpec, max_pos: int, device="cuda") -> torch.Tensor:
    """RoPE table built by the library on the device (gqa_rope_table_build)."""
    w = gqa.gqa_rope_inv_freq(d, rope.base, rope.yarn_factor, rope.yarn_L0, rope.beta_fast,
                              rope.beta_slow, rope.rotate_fraction)
    tab = torch.empty(max_pos * (d // 2) * 2, dtype=torch.float32, device=device)
    gqa.gqa_rope_table_build(tab, w, d, rope.amp, max_pos)
    return tab


def oracle_freq(d: int, rope: RopeSpec) -> np.ndarray:
    return orc().inv_freq(d, rope.base, rope.yarn_factor, rope.yarn_L0, rope.beta_fast,
                          rope.beta_slow, rope.rotate_fraction)


def run_prefill(q, k, v, window: int, scale: float, table: torch.Tensor, table_len: int,
                want_lse: bool = True, k_mode: int = 0):
    """q/k/v on the GPU (bf16), k before RoPE.  Returns (o, lse) from gqa_attn_prefill;
    k_mode is its k_is_rotated argument: 0 rotates K once into a workspace, 2 rotates each
    K tile inside the attention kernel."""
    B, Hq, T, d = q.shape
    _, Hkv, S, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device) if want_lse else None
    wsb = gqa.gqa_prefill_workspace_bytes(B, Hkv, S, d) if k_mode == 0 else 0
    ws = torch.empty(wsb, dtype=torch.uint8, device=q.device) if wsb else None
    gqa.gqa_attn_prefill(q, k, v, o, lse, B, T, S, Hq, Hkv, d, window, scale, table,
                         table_len, k_mode, ws, wsb)
    st = gqa.gqa_get_device_status()
    assert st == 0, f"device status {gqa.STATUS_NAMES.get(st, st)}"
    return o, lse


def compare(gpu: torch.Tensor, ref: np.ndarray, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    mx, mn = float(err.max()), float(err.mean())
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max abs {mx:.3e}, mean abs {mn:.3e}"
    return mx, mn


def sample_rows(B: int, Hq: int, Hkv: int, T: int, window: int, n_target: int, seed: int):
    """(b, h, t) rows for sampled parity: every head of two KV groups (first and last)
    plus random rows; always the edge positions 0, 1, W-2, W-1, W, multiples of 128 +- 1,
    and T-1."""
    rng = np.random.default_rng(seed)
    G = Hq // Hkv
    heads = sorted(set(list(range(G)) + list(range((Hkv - 1) * G, Hkv * G))))
    edges = {0, 1, T - 1, T - 2}
    if window > 0:
        edges |= {window - 2, window - 1, window, window + 1}
    for m in range(128, T, 128 * max(1, T // 2048)):
        edges |= {m - 1, m, m + 1}
    edges = sorted(t for t in edges if 0 <= t < T)
    rows = set()
    for b in range(B):
        for h in heads:
            for t in edges:
                rows.add((b, h, t))
    while len(rows) < n_target:
        rows.add((int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(T))))
    return np.array(sorted(rows), dtype=np.int32)


def to_cuda(*ts):
    return [t.cuda() for t in ts]
