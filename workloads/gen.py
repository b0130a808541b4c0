"""Seeded random draws for the workloads (no attention arithmetic here).

All draws use torch's CPU generator so that the same seed gives the same bits on
x86 and on Arm hosts.  Tensors are returned on the CPU; callers move them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List

import numpy as np
import torch

from .configs import DecodeWorkload, PrefillLayer, RopeSpec


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, seed: int) -> torch.Tensor:
    """N(0, 1) float32 draws rounded once to bfloat16 (round to nearest even)."""
    return torch.randn(*shape, generator=_gen(seed), dtype=torch.float32).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bfloat16 bit patterns of a CPU tensor, as a contiguous uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class PrefillInputs:
    q: torch.Tensor   # [B, Hq, T, d] bf16
    k: torch.Tensor   # [B, Hkv, S, d] bf16, before RoPE (as a cache holds it)
    v: torch.Tensor   # [B, Hkv, S, d] bf16


def prefill_inputs(layer: PrefillLayer) -> PrefillInputs:
    s = layer.seed * 16
    q = randn_bf16((layer.B, layer.Hq, layer.T, layer.d), s + 1)
    k = randn_bf16((layer.B, layer.Hkv, layer.S, layer.d), s + 2)
    v = randn_bf16((layer.B, layer.Hkv, layer.S, layer.d), s + 3)
    return PrefillInputs(q, k, v)


@dataclass
class DecodeInputs:
    q: torch.Tensor              # [nseq, Hq, d] bf16 (the one new query token per sequence)
    k_new: torch.Tensor          # [nseq, Hkv, d] bf16 (the new token's key, before RoPE)
    v_new: torch.Tensor          # [nseq, Hkv, d] bf16
    k_cache: List[torch.Tensor]  # per sequence [Hkv, cap, d] bf16, slots as stored
    v_cache: List[torch.Tensor]
    cap: List[int]               # slots per (sequence, KV head)
    count_before: List[int]      # linear cache: tokens held; ring: tokens ever appended
    is_ring: List[int]
    rope: List[RopeSpec]


def decode_inputs(w: DecodeWorkload, cap_slack: int = 0) -> DecodeInputs:
    """Draws one decode batch.

    Global sequences: total length after the append S ~ U{lo..hi} (inclusive), so the
    cache holds S - 1 tokens beforehand; capacity S + cap_slack.
    Local sequences: a ring of capacity `w.window`; the count of tokens appended so far
    is drawn from [window - 1, window - 1 + 4 * window) so the next write slot falls
    anywhere in the ring.
    """
    base = w.seed * 16
    nseq = w.nseq
    q = randn_bf16((nseq, w.Hq, w.d), base + 1)
    k_new = randn_bf16((nseq, w.Hkv, w.d), base + 2)
    v_new = randn_bf16((nseq, w.Hkv, w.d), base + 3)
    lo, hi = w.global_len_range
    g_len = torch.randint(lo, hi + 1, (w.n_global,), generator=_gen(base + 4)).tolist()
    r_cnt = torch.randint(w.window - 1, w.window - 1 + 4 * w.window, (w.n_local,),
                          generator=_gen(base + 5)).tolist()
    k_cache, v_cache, cap, count, ring, rope = [], [], [], [], [], []
    for i in range(nseq):
        if i < w.n_global:
            S = int(g_len[i])
            c = S + cap_slack
            count.append(S - 1)
            ring.append(0)
            rope.append(w.rope_global)
        else:
            c = w.window
            count.append(int(r_cnt[i - w.n_global]))
            ring.append(1)
            rope.append(w.rope_local)
        cap.append(c)
        k_cache.append(randn_bf16((w.Hkv, c, w.d), base + 100 + 2 * i))
        v_cache.append(randn_bf16((w.Hkv, c, w.d), base + 101 + 2 * i))
    return DecodeInputs(q, k_new, v_new, k_cache, v_cache, cap, count, ring, rope)


def norm_gains(d: int, seed: int) -> np.ndarray:
    """A per-layer RMSNorm gain [d] for a layer with attention scale 1 (Gemma 4): values
    around d^(-1/4) with 20% spread, so a query/key gain pair gives logits of standard
    deviation ~1 on unit-RMS rows (what scale 1/sqrt(d) gives the other workloads).
    Rounded to bf16 values (as stored weights are), returned as float64."""
    g = torch.randn(d, generator=_gen(seed), dtype=torch.float32)
    level = d ** -0.25
    return (level * (1.0 + 0.2 * g)).to(torch.bfloat16).to(torch.float64).numpy()
