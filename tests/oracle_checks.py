"""Pins for the fp64 oracle: each check raises AssertionError when the oracle is wrong.

Every check compares the oracle with something other than itself: a value the pages
print, a closed form, a library routine (torch SDPA, numpy complex arithmetic), brute
force, or an invariant of the mathematics.  `tests/test_oracle_pins.py` runs them on
the oracle; `tests/test_oracle_planted.py` runs them on builds with a planted mistake
and requires that at least one check fails for each.
"""
from __future__ import annotations

import json
import math
import os
from collections import deque

import numpy as np
import torch

from oracle import twin

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------------
# printed values
# ---------------------------------------------------------------------------------

def check_worked_example(orc):
    """Values printed for the three-token example (troy-technical.jp explainer, §4, Fig. 3)."""
    g = _golden("worked_example_attention.json")
    q = torch.tensor(g["Q"], dtype=torch.bfloat16).reshape(1, 1, 3, 2)
    k = torch.tensor(g["K"], dtype=torch.bfloat16).reshape(1, 1, 3, 2)
    v = torch.tensor(g["V"], dtype=torch.bfloat16).reshape(1, 1, 3, 2)
    o, _, wts = orc.attention(q, k, v, window=0, scale=math.sqrt(g["scale_sq"]),
                              w=np.zeros(1), amp=1.0, want_weights=True)
    tol = g["tolerance"]
    for t, row in enumerate(g["weights"]):
        for s, val in enumerate(row):
            assert abs(wts[0, 0, t, s] - val) <= tol, (t, s, wts[0, 0, t, s], val)
        assert np.all(wts[0, 0, t, len(row):] == 0.0)
    assert np.max(np.abs(o[0, 0] - np.array(g["outputs"]))) <= tol, o[0, 0]


def check_yarn_constants(orc):
    """YaRN boundaries and amplitude printed in "PLaMo 3アーキテクチャ徹底解析" §6.3."""
    g = _golden("yarn_constants.json")
    jl = orc.yarn_boundary(g["d"], g["base"], g["L0"], g["beta_fast"])
    jh = orc.yarn_boundary(g["d"], g["base"], g["L0"], g["beta_slow"])
    assert abs(jl - g["j_low"]) <= g["tol_boundary"], jl
    assert abs(jh - g["j_high"]) <= g["tol_boundary"], jh
    a = orc.yarn_amp(g["s"])
    assert abs(a - g["amp"]) <= g["tol_amp"], a
    assert abs(a * a - g["amp_sq"]) <= g["tol_amp"], a * a
    assert abs(a * a / math.sqrt(g["d"]) - g["amp_sq_over_sqrt_d"]) <= g["tol_amp"]


def check_yarn_curve(orc):
    """Fig. 7 of §6.3: multiplier 1 up to the low boundary, 1/s from the high one, a
    straight line between them, boundaries used unrounded."""
    g = _golden("yarn_constants.json")
    d, base, s = g["d"], g["base"], g["s"]
    plain = orc.inv_freq(d, base)
    yarn = orc.inv_freq(d, base, yarn_factor=s, yarn_L0=g["L0"], beta_fast=g["beta_fast"],
                        beta_slow=g["beta_slow"])
    ratio = yarn / plain
    assert np.all(ratio[:14] == 1.0), ratio[:14]                   # j <= 13 < 13.96
    assert np.allclose(ratio[31:], 1.0 / s, rtol=1e-14, atol=0)   # j >= 31 > 30.02
    mid = ratio[14:31]
    assert np.all(np.diff(mid) < 0)
    # linear in j strictly between the boundaries: zero second differences
    assert np.max(np.abs(np.diff(ratio[14:31], 2))) < 1e-13
    # unrounded boundaries: j = 14 already interpolates, j = 30 is not yet at 1/s
    assert ratio[14] < 1.0 and ratio[30] > 1.0 / s
    # the line through the interior hits 1 at ~13.96 and 1/s at ~30.02
    slope = ratio[15] - ratio[14]
    j_at_one = 14 - (1.0 - ratio[14]) / (-slope)
    j_at_min = 14 + (ratio[14] - 1.0 / s) / (-slope)
    assert abs(j_at_one - g["j_low"]) < g["tol_boundary"], j_at_one
    assert abs(j_at_min - g["j_high"]) < g["tol_boundary"], j_at_min


def check_base_frequencies(orc):
    """§6.1: omega_j = theta^(-2j/d): omega_0 = 1 (wavelength 2 pi tokens), omega_{d/4} =
    theta^(-1/2), strictly decreasing, lowest at j = d/2 - 1."""
    for d, base in ((128, 1e4), (128, 1e6), (256, 1e4), (16, 1e4)):
        w = orc.inv_freq(d, base)
        assert w.shape == (d // 2,)
        assert w[0] == 1.0
        assert abs(w[d // 4] - base ** -0.5) <= 1e-15 * max(1.0, base ** -0.5)
        assert np.all(np.diff(w) < 0)
        assert abs(w[-1] - base ** (-(d - 2) / d)) <= 1e-15


def check_p_rope(orc):
    """§6.4: head dim 512, p = 0.25: pairs 0..63 rotate with (1e6)^(-2j/512), pairs 64..255
    have frequency 0; only components 0..63 and 256..319 change."""
    w = orc.inv_freq(512, 1e6, rotate_fraction=0.25)
    assert np.all(w[64:] == 0.0)
    assert abs(w[63] - 1e6 ** (-126 / 512)) < 1e-16 and w[0] == 1.0
    x = _f64(_bf16((512,), 11))
    y = orc.rope_rotate(x, 1234.0, w, 1.0)
    changed = np.nonzero(y != x)[0]
    assert set(changed.tolist()) == set(range(64)) | set(range(256, 320)), changed


def check_rope_complex(orc):
    """§6.1 rotation of the pair (x_j, x_{j+d/2}) by angle p omega_j, against numpy's
    complex multiplication (a + ib) amp e^{i p omega}; norm scales by amp."""
    d = 128
    w = orc.inv_freq(d, 1e4)
    rng = np.random.default_rng(5)
    for pos in (0, 1, 7, 2047, 65535):
        x = rng.standard_normal(d)
        for amp in (1.0, 1.5545):
            y = orc.rope_rotate(x, pos, w, amp)
            z = (x[:64] + 1j * x[64:]) * amp * np.exp(1j * pos * w)
            assert np.max(np.abs(y[:64] - z.real)) < 1e-12
            assert np.max(np.abs(y[64:] - z.imag)) < 1e-12
            assert abs(np.linalg.norm(y) - amp * np.linalg.norm(x)) < 1e-11
    # a unit vector on pair 3 lands on (cos, sin) of its angle
    e = np.zeros(d)
    e[3] = 1.0
    y = orc.rope_rotate(e, 5.0, w, 1.0)
    assert abs(y[3] - math.cos(5 * w[3])) < 1e-15 and abs(y[67] - math.sin(5 * w[3])) < 1e-15


def check_relative_position(orc):
    """RoPE property the pages use (§4.4; LLaMA tutorial, RoPE properties): the rotated dot
    product depends on the position difference only."""
    d = 128
    w = orc.inv_freq(d, 1e6, yarn_factor=8.0)
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    ref = orc.rope_rotate(q, 100, w, 1.2) @ orc.rope_rotate(k, 37, w, 1.2)
    for shift in (1, 1000, 60000):
        val = orc.rope_rotate(q, 100 + shift, w, 1.2) @ orc.rope_rotate(k, 37 + shift, w, 1.2)
        assert abs(val - ref) < 1e-9 * max(1.0, abs(ref)), (shift, val, ref)


# ---------------------------------------------------------------------------------
# attention against a library routine and brute force
# ---------------------------------------------------------------------------------

def _sdpa(q, k, v, window, scale):
    """torch's scaled_dot_product_attention in fp64 on the CPU with an explicit boolean
    mask and enable_gqa (the routine the public implementation calls, §4.2)."""
    B, Hq, T, d = q.shape
    S = k.shape[2]
    i = torch.arange(S - T, S)[:, None]
    j = torch.arange(S)[None, :]
    allowed = j <= i
    if window > 0:
        allowed &= (i - j) < window
    return torch.nn.functional.scaled_dot_product_attention(
        q.to(torch.float64), k.to(torch.float64), v.to(torch.float64),
        attn_mask=allowed, scale=scale, enable_gqa=True).numpy()


def check_sdpa_no_rope(orc):
    """With all frequencies 0 and amp 1 the rotation is the identity (§6.4), so the oracle
    must equal torch SDPA (fp64, boolean mask, GQA) to rounding."""
    cases = [(1, 6, 6, 4, 2, 16, 0), (2, 5, 9, 6, 3, 8, 3), (1, 12, 12, 8, 2, 32, 4),
             (1, 7, 7, 2, 1, 4, 1), (1, 16, 16, 4, 4, 8, 20)]
    for n, (B, T, S, Hq, Hkv, d, W) in enumerate(cases):
        q = _bf16((B, Hq, T, d), 100 + n)
        k = _bf16((B, Hkv, S, d), 200 + n)
        v = _bf16((B, Hkv, S, d), 300 + n)
        scale = 1.0 / math.sqrt(d)
        o, _ = orc.attention(q, k, v, window=W, scale=scale, w=np.zeros(d // 2), amp=1.0)
        ref = _sdpa(q, k, v, W, scale)
        assert np.max(np.abs(o - ref)) < 1e-12, (n, np.max(np.abs(o - ref)))


def check_twin_brute_force(orc):
    """Against the dense numpy twin (complex-number RoPE, np.repeat GQA), with YaRN
    frequencies, amplitude, windows and a position shift."""
    cases = [
        (1, 9, 9, 4, 2, 16, 0, dict(base=1e4), 1.0, 0),
        (2, 7, 11, 6, 2, 8, 4, dict(base=1e6, yarn_factor=8.0), math.sqrt(1.2), 0),
        (1, 13, 13, 8, 1, 32, 5, dict(base=1e4), 1.0, 17),
        (1, 10, 10, 4, 4, 16, 0, dict(base=1e6, rotate_fraction=0.25), 1.0, 0),
        (1, 5, 5, 2, 1, 64, 1, dict(base=1e4), 1.0, 0),
    ]
    for n, (B, T, S, Hq, Hkv, d, W, rs, amp, shift) in enumerate(cases):
        q = _bf16((B, Hq, T, d), 400 + n)
        k = _bf16((B, Hkv, S, d), 500 + n)
        v = _bf16((B, Hkv, S, d), 600 + n)
        scale = 1.0 / math.sqrt(d)
        w = orc.inv_freq(d, **rs)
        wt = twin.inv_freq(d, **rs)
        assert np.max(np.abs(w - wt)) < 1e-15, (n, "frequencies")
        o, lse = orc.attention(q, k, v, window=W, scale=scale, w=w, amp=amp, pos_shift=shift)
        ot, lset = twin.attention(_f64(q), _f64(k), _f64(v), W, scale, wt, amp, shift)
        assert np.max(np.abs(o - ot)) < 1e-12, (n, np.max(np.abs(o - ot)))
        assert np.max(np.abs(lse - lset)) < 1e-12, n


# ---------------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------------

def check_window_ge_T_is_global(orc):
    """§5.1: a window at least T wide removes nothing, so the result equals full causal."""
    q, k, v = _bf16((1, 4, 20, 16), 701), _bf16((1, 2, 20, 16), 702), _bf16((1, 2, 20, 16), 703)
    w = orc.inv_freq(16, 1e4)
    og, _ = orc.attention(q, k, v, window=0, scale=0.25, w=w, amp=1.0)
    for W in (20, 21, 1000):
        ow, _ = orc.attention(q, k, v, window=W, scale=0.25, w=w, amp=1.0)
        assert np.array_equal(og, ow)
    o19, _ = orc.attention(q, k, v, window=19, scale=0.25, w=w, amp=1.0)
    assert not np.array_equal(og, o19)


def check_weights_rows(orc):
    """Softmax rows sum to 1; masked keys (future, or i - j >= W) get weight exactly 0."""
    T, W = 24, 5
    q, k, v = _bf16((1, 2, T, 16), 801), _bf16((1, 1, T, 16), 802), _bf16((1, 1, T, 16), 803)
    w = orc.inv_freq(16, 1e4)
    _, _, wts = orc.attention(q, k, v, window=W, scale=0.25, w=w, amp=1.0, want_weights=True)
    assert np.max(np.abs(wts.sum(-1) - 1.0)) < 1e-12
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    visible = (j <= i) & (i - j < W)
    assert np.all(wts[..., ~visible] == 0.0)
    assert np.all(wts[..., visible] > 0.0)
    # the window counts self: row 10 sees exactly keys 6..10
    assert np.nonzero(wts[0, 0, 10])[0].tolist() == [6, 7, 8, 9, 10]


def check_shift_invariance(orc):
    """§4.4: shifting every Q and K position by the same amount leaves the scores unchanged
    up to rounding (the reason the local cache may re-number positions from 0)."""
    q, k, v = _bf16((1, 4, 12, 32), 901), _bf16((1, 2, 12, 32), 902), _bf16((1, 2, 12, 32), 903)
    for rs, amp in ((dict(base=1e4), 1.0), (dict(base=1e6, yarn_factor=8.0), math.sqrt(1.2))):
        w = orc.inv_freq(32, **rs)
        o0, _ = orc.attention(q, k, v, window=6, scale=0.2, w=w, amp=amp)
        for shift in (3, 2047, 50000):
            o1, _ = orc.attention(q, k, v, window=6, scale=0.2, w=w, amp=amp, pos_shift=shift)
            assert np.max(np.abs(o1 - o0)) < 1e-9, (shift, np.max(np.abs(o1 - o0)))


def check_gqa_grouping(orc):
    """§4.2: consecutive query heads share a KV head.  Changing KV head 1 changes exactly
    query heads G..2G-1; permuting heads inside a group permutes their outputs."""
    Hq, Hkv, d, T = 6, 3, 16, 8
    G = Hq // Hkv
    q, k, v = _bf16((1, Hq, T, d), 1001), _bf16((1, Hkv, T, d), 1002), _bf16((1, Hkv, T, d), 1003)
    w = orc.inv_freq(d, 1e4)
    o0, _ = orc.attention(q, k, v, window=0, scale=0.25, w=w, amp=1.0)
    v2 = v.clone()
    v2[:, 1] = _bf16((T, d), 1004)
    o1, _ = orc.attention(q, k, v2, window=0, scale=0.25, w=w, amp=1.0)
    changed = [h for h in range(Hq) if not np.array_equal(o0[0, h], o1[0, h])]
    assert changed == list(range(G, 2 * G)), changed
    perm = [1, 0, 2, 3, 5, 4]
    op, _ = orc.attention(q[:, perm], k, v, window=0, scale=0.25, w=w, amp=1.0)
    assert np.array_equal(op[0], o0[0, perm])
    for h in range(Hq):
        assert orc.kv_head(h, Hq, Hkv) == h // G == (h * Hkv) // Hq


def check_cache_index_bruteforce(orc):
    """§4.4 cache model against a simulation: a slot array written token by token, and a
    list that keeps only the newest W-1 tokens after each step (the local cache)."""
    for W in (1, 2, 3, 4, 5, 8, 64):
        slots = [None] * W
        kept = deque()
        for n in range(0, 5 * W + 3):       # n = tokens appended before this step
            s = orc.append_slot(1, n, W)
            assert s == n % W
            slots[s] = n                     # token id n written
            kept.append(n)                   # the W-1 kept plus the new one
            R = orc.retained(1, n + 1, W)
            assert R == len(kept) == min(n + 1, W)
            for t in range(R):
                assert slots[orc.logical_slot(1, n + 1, W, t)] == kept[t], (W, n, t)
            while len(kept) > W - 1:
                kept.popleft()
    for cap in (1, 5, 100):
        for n in range(cap + 2):
            s = orc.append_slot(0, n, cap)
            assert s == (n if n < cap else -1)
            if s >= 0:
                assert orc.retained(0, n + 1, cap) == n + 1
                assert all(orc.logical_slot(0, n + 1, cap, t) == t for t in range(n + 1))


def _decode_case(orc, seed, is_ring, count_before, cap, Hq=4, Hkv=2, d=16, base=1e4, amp=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(1, Hq, d, generator=g).to(torch.bfloat16)
    kn = torch.randn(1, Hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(1, Hkv, d, generator=g).to(torch.bfloat16)
    kc = torch.randn(Hkv, cap, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(Hkv, cap, d, generator=g).to(torch.bfloat16)
    w = orc.inv_freq(d, base)
    o, lse, slots, after = orc.decode_step(q, kn, vn, [kc], [vc], [cap], [count_before],
                                           [is_ring], [w], [amp], 0.25)
    return q, kn, vn, kc, vc, w, o, slots, after


def check_decode_equals_prefill_row(orc):
    """§10 check "batch vs token-by-token decode": decoding with a linear cache holding
    tokens 0..t-1 gives row t of prefill over tokens 0..t."""
    Hq, Hkv, d, t = 4, 2, 16, 9
    q, kn, vn, kc, vc, w, o, slots, after = _decode_case(orc, 1101, 0, t, t + 3)
    assert slots[0] == t and after[0] == t + 1
    K = torch.cat([kc[:, :t], kn[0][:, None]], dim=1)[None]
    V = torch.cat([vc[:, :t], vn[0][:, None]], dim=1)[None]
    Q = torch.zeros(1, Hq, t + 1, d, dtype=torch.bfloat16)
    Q[0, :, t] = q[0]
    op, _ = orc.attention(Q, K, V, window=0, scale=0.25, w=w, amp=1.0)
    assert np.max(np.abs(op[0, :, t] - o[0])) < 1e-12


def check_ring_equals_full_history(orc):
    """§4.4: the ring (last W-1 kept, +1 new, re-numbered 0..W-1) equals windowed attention
    over the full history at absolute positions, up to rounding."""
    W, Hq, Hkv, d = 6, 4, 2, 16
    for n_before in (W - 1, W + 2, 4 * W + 1):
        g = torch.Generator().manual_seed(1200 + n_before)
        hist_k = torch.randn(Hkv, n_before + 1, d, generator=g).to(torch.bfloat16)
        hist_v = torch.randn(Hkv, n_before + 1, d, generator=g).to(torch.bfloat16)
        q = torch.randn(1, Hq, d, generator=g).to(torch.bfloat16)
        ring_k = torch.zeros(Hkv, W, d, dtype=torch.bfloat16)
        ring_v = torch.zeros(Hkv, W, d, dtype=torch.bfloat16)
        for i in range(n_before):            # tokens 0..n_before-1 written slot i mod W
            ring_k[:, i % W] = hist_k[:, i]
            ring_v[:, i % W] = hist_v[:, i]
        w = orc.inv_freq(d, 1e4)
        o, _, _, _ = orc.decode_step(q, hist_k[:, n_before][None], hist_v[:, n_before][None],
                                     [ring_k], [ring_v], [W], [n_before], [1], [w], [1.0], 0.3)
        Q = torch.zeros(1, Hq, n_before + 1, d, dtype=torch.bfloat16)
        Q[0, :, n_before] = q[0]
        of, _ = orc.attention(Q, hist_k[None], hist_v[None], window=W, scale=0.3, w=w, amp=1.0)
        assert np.max(np.abs(of[0, :, n_before] - o[0])) < 1e-9, n_before


# ---------------------------------------------------------------------------------
# RMSNorm with an effective gain (PLaMo page §3.2 formula, §4.3 q_norm / k_norm)
# ---------------------------------------------------------------------------------

def check_rms_norm_closed_form(orc):
    """A constant vector a*1 normalises to gamma * a / sqrt(a^2 + eps) in every
    component; with eps = 0 any vector's normalised mean square (gain 1) is exactly 1."""
    n, a, eps = 128, 2.0, 1e-6
    x = torch.full((2, n), a).to(torch.bfloat16)
    gamma = 1.0 + np.linspace(-0.25, 0.5, n)          # offset 1 plus a stored weight
    y = orc.rms_norm(x, gamma, eps)
    want = gamma * a / math.sqrt(a * a + eps)
    assert np.max(np.abs(y - want[None, :])) < 1e-12, np.max(np.abs(y - want))
    z = orc.rms_norm(_bf16((5, 96), 501), None, 0.0)
    assert np.max(np.abs(np.mean(z * z, axis=-1) - 1.0)) < 1e-12


def check_rms_norm_library(orc):
    """torch.nn.functional.rms_norm in fp64 with the effective gain as its weight."""
    x = _bf16((7, 3, 128), 502)
    gamma = 1.0 + 0.1 * _f64(_bf16((128,), 503))
    y = orc.rms_norm(x, gamma, 1e-6)
    ref = torch.nn.functional.rms_norm(x.to(torch.float64), (128,),
                                       weight=torch.from_numpy(gamma), eps=1e-6).numpy()
    assert np.max(np.abs(y - ref)) < 1e-12, np.max(np.abs(y - ref))


def check_rms_norm_scale_invariance(orc):
    """N(4x) = N(x) up to the epsilon term (4x is exact in bf16)."""
    x = _bf16((6, 128), 504)
    x4 = (x.to(torch.float32) * 4).to(torch.bfloat16)
    a = orc.rms_norm(x, None, 1e-6)
    b = orc.rms_norm(x4, None, 1e-6)
    assert np.max(np.abs(a - b)) < 1e-5, np.max(np.abs(a - b))


# ---------------------------------------------------------------------------------
# shared K/V projection (attention_k_eq_v of Gemma 4's global layers: PLaMo page §5.2
# and §8 -- K = RoPE(N_{gamma_k}(Z)), V = N_1(Z))
# ---------------------------------------------------------------------------------

def _gains(d, seed, level):
    g = torch.Generator().manual_seed(seed)
    return level * (1.0 + 0.2 * torch.randn(d, generator=g, dtype=torch.float64)).numpy()


def check_kv_shared_library(orc):
    """Against torch.nn.functional.rms_norm (fp64) for the three norms -- gain gamma_q on
    the query, gamma_k on the keys, none on the values -- followed by the numpy twin's
    attention (complex-number RoPE, dense softmax)."""
    cases = [(1, 7, 7, 4, 2, 16, 0, dict(base=1e4), 1.0),
             (1, 5, 9, 4, 1, 32, 4, dict(base=1e6, rotate_fraction=0.25), 1.0),
             (2, 6, 6, 6, 3, 8, 3, dict(base=1e6, yarn_factor=8.0), math.sqrt(1.2))]
    eps = 1e-6
    for n, (B, T, S, Hq, Hkv, d, W, rs, amp) in enumerate(cases):
        q = _bf16((B, Hq, T, d), 700 + n)
        z = (_bf16((B, Hkv, S, d), 710 + n).to(torch.float32) * 3).to(torch.bfloat16)
        gq, gk = _gains(d, 720 + n, 0.6), _gains(d, 730 + n, 0.6)
        w = orc.inv_freq(d, **rs)
        o, lse = orc.attention_kv_shared(q, z, q_gamma=gq, k_gamma=gk, eps=eps, window=W,
                                         scale=1.0, w=w, amp=amp)
        rn = torch.nn.functional.rms_norm
        qn = rn(q.to(torch.float64), (d,), weight=torch.from_numpy(gq), eps=eps).numpy()
        kn = rn(z.to(torch.float64), (d,), weight=torch.from_numpy(gk), eps=eps).numpy()
        vn = rn(z.to(torch.float64), (d,), eps=eps).numpy()
        ot, lset = twin.attention(qn, kn, vn, W, 1.0, twin.inv_freq(d, **rs), amp)
        assert np.max(np.abs(o - ot)) < 1e-12, (n, np.max(np.abs(o - ot)))
        assert np.max(np.abs(lse - lset)) < 1e-12, n


def check_kv_shared_decode(orc):
    """Decode of a shared-projection layer: with a linear cache of Z holding tokens
    0..t-1 it gives row t of the prefill over tokens 0..t; with a ring (last W-1 kept plus
    the new token, re-numbered) it gives windowed attention over the whole history."""
    Hq, Hkv, d, eps = 4, 2, 16, 1e-6
    gq, gk = _gains(d, 740, 0.7), _gains(d, 741, 0.7)
    w = orc.inv_freq(d, 1e4)
    for is_ring, n_before, cap in ((0, 9, 12), (1, 5, 6), (1, 15, 6), (1, 25, 6)):
        g = torch.Generator().manual_seed(750 + n_before + 100 * is_ring)
        hist = torch.randn(Hkv, n_before + 1, d, generator=g).to(torch.bfloat16)
        q = torch.randn(1, Hq, d, generator=g).to(torch.bfloat16)
        cache = torch.randn(Hkv, cap, d, generator=g).to(torch.bfloat16)   # stale slots
        for i in range(n_before):
            cache[:, i % cap if is_ring else i] = hist[:, i]
        o, _, slots, after = orc.decode_step_kv_shared(
            q, hist[:, n_before][None], [cache], [cap], [n_before], [is_ring], [w], [1.0],
            q_gamma=gq, k_gamma=gk, eps=eps, scale=0.5)
        assert slots[0] == (n_before % cap if is_ring else n_before)
        assert after[0] == n_before + 1
        Q = torch.zeros(1, Hq, n_before + 1, d, dtype=torch.bfloat16)
        Q[0, :, n_before] = q[0]
        of, _ = orc.attention_kv_shared(Q, hist[None], q_gamma=gq, k_gamma=gk, eps=eps,
                                        window=cap if is_ring else 0, scale=0.5, w=w, amp=1.0)
        assert np.max(np.abs(of[0, :, n_before] - o[0])) < 1e-9, (is_ring, n_before)


ALL_CHECKS = [
    check_kv_shared_library,
    check_kv_shared_decode,
    check_rms_norm_closed_form,
    check_rms_norm_library,
    check_rms_norm_scale_invariance,
    check_worked_example,
    check_yarn_constants,
    check_yarn_curve,
    check_base_frequencies,
    check_p_rope,
    check_rope_complex,
    check_relative_position,
    check_sdpa_no_rope,
    check_twin_brute_force,
    check_window_ge_T_is_global,
    check_weights_rows,
    check_shift_invariance,
    check_gqa_grouping,
    check_cache_index_bruteforce,
    check_decode_equals_prefill_row,
    check_ring_equals_full_history,
]
