"""Dense numpy fp64 twin of the oracle, for tiny brute-force cross-checks.

TEST INFRASTRUCTURE (see the package docstring).  Written independently of
``gqa_oracle.c`` in a different formulation: the split-half rotation is a complex
multiplication (a + i b) * amp * exp(i p omega_j); GQA is `np.repeat` of the KV heads;
the mask is a dense boolean matrix; the softmax is over a dense score matrix.  It
follows "PLaMo 3アーキテクチャ徹底解析" §4.2, §4.4, §4.5, §5.1, §6.1, §6.3, §6.4.
Use only on tiny shapes: it materialises every score.
"""
from __future__ import annotations

import numpy as np


def inv_freq(d: int, base: float, yarn_factor: float = 1.0, yarn_L0: float = 4096.0,
             beta_fast: float = 32.0, beta_slow: float = 1.0,
             rotate_fraction: float = 1.0) -> np.ndarray:
    j = np.arange(d // 2, dtype=np.float64)
    om = np.power(base, -2.0 * j / d)
    if yarn_factor != 1.0:
        def boundary(beta):
            return (d / 2) * np.log(yarn_L0 / (2 * np.pi * beta)) / np.log(base)
        lo, hi = boundary(beta_fast), boundary(beta_slow)
        alpha = np.clip((j - lo) / (hi - lo), 0.0, 1.0)
        om = om * (1.0 - alpha) + (om / yarn_factor) * alpha
    if rotate_fraction < 1.0:
        om = np.where(j >= np.floor(rotate_fraction * (d // 2) + 0.5), 0.0, om)
    return om


def rope(x: np.ndarray, pos: np.ndarray, om: np.ndarray, amp: float) -> np.ndarray:
    """x [..., n, d] at positions pos [n]; pair j is the complex number x_j + i x_{j+d/2}."""
    half = x.shape[-1] // 2
    z = x[..., :half] + 1j * x[..., half:]
    z = z * (amp * np.exp(1j * np.outer(pos.astype(np.float64), om)))
    return np.concatenate([z.real, z.imag], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, window: int, scale: float,
              om: np.ndarray, amp: float, pos_shift: int = 0):
    """q [B,Hq,T,d], k/v [B,Hkv,S,d] as float64.  Returns (o [B,Hq,T,d], lse [B,Hq,T])."""
    B, Hq, T, d = q.shape
    S, Hkv = k.shape[2], k.shape[1]
    qpos = np.arange(S - T, S)
    kpos = np.arange(S)
    qr = rope(q, qpos + pos_shift, om, amp)
    kr = np.repeat(rope(k, kpos + pos_shift, om, amp), Hq // Hkv, axis=1)
    vv = np.repeat(v, Hq // Hkv, axis=1)
    scores = np.einsum("bhtd,bhsd->bhts", qr, kr) * scale
    diff = qpos[:, None] - kpos[None, :]
    allowed = diff >= 0
    if window > 0:
        allowed &= diff < window
    scores = np.where(allowed, scores, -np.inf)
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    l = e.sum(axis=-1, keepdims=True)
    return np.einsum("bhts,bhsd->bhtd", e / l, vv), (m + np.log(l))[..., 0]
