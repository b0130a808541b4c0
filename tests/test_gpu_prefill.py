"""Prefill parity: gqa_attn_prefill (C-ABI, tcgen05 kernel) against the fp64 oracle.

Small cases compare every output element; the full-size PLaMo-3-shaped workloads
(same launch configuration the benchmark times) compare a seeded sample of rows that
always includes the window edges, tile edges and the last row.  Bar: max abs 2e-2 and
mean abs 2e-3 on the bf16 outputs; lse within 2e-2.
"""
import math

import numpy as np
import pytest
import torch

import gpu_utils as gu
from workloads import WORKLOADS, PrefillLayer, RopeSpec, prefill_inputs

pytestmark = pytest.mark.gpu

LOCAL = RopeSpec(base=1e4)
YARN = RopeSpec(base=1e6, yarn_factor=8.0, amp=math.sqrt(1.2))


def _full_case(layer: PrefillLayer):
    gu.require_gpu()
    x = prefill_inputs(layer)
    q, k, v = gu.to_cuda(x.q, x.k, x.v)
    table = gu.rope_table(layer.d, layer.rope, layer.S)
    o, lse = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S)
    w = gu.oracle_freq(layer.d, layer.rope)
    ro, rl = gu.orc().attention(x.q, x.k, x.v, window=layer.window, scale=layer.scale, w=w,
                                amp=layer.rope.amp)
    gu.compare(o, ro, what=layer.label)
    gu.compare(lse, rl, max_abs=2e-2, mean_abs=2e-3, what=layer.label + " lse")
    return o


@pytest.mark.parametrize("name", ["tiny_w64", "tiny_causal"])
def test_tiny_workloads(name):
    _full_case(WORKLOADS[name].layers[0])


def _layer(B, T, S, Hq, Hkv, W, rope=LOCAL, seed=7, d=128):
    return PrefillLayer(B=B, T=T, S=S, Hq=Hq, Hkv=Hkv, d=d, window=W, rope=rope,
                        scale=1 / math.sqrt(d), seed=seed)


EDGE_CASES = [
    # ragged tails, several tiles, tiny windows, windows at tile edges
    _layer(1, 200, 200, 2, 1, 0, seed=11),
    _layer(1, 1, 1, 2, 1, 0, seed=12),
    _layer(1, 130, 130, 4, 2, 1, seed=13),
    _layer(1, 300, 300, 4, 1, 4, seed=14),
    _layer(1, 384, 384, 2, 1, 127, seed=15),
    _layer(1, 384, 384, 2, 1, 128, seed=16),
    _layer(1, 384, 384, 2, 1, 129, seed=17),
    _layer(2, 257, 257, 6, 2, 64, YARN, seed=18),
    # odd group (last head pair has one head), MHA, MQA
    _layer(1, 160, 160, 3, 1, 0, seed=19),
    _layer(1, 160, 160, 2, 2, 50, seed=20),
    _layer(1, 256, 256, 8, 1, 0, YARN, seed=21),
    # queries at the end of a longer key range (chunked prefill: q_pos = S - T + t)
    _layer(1, 100, 300, 4, 2, 0, seed=22),
    _layer(1, 129, 700, 4, 2, 200, YARN, seed=23),
    _layer(1, 1, 513, 2, 1, 0, seed=24),
]


@pytest.mark.parametrize("layer", EDGE_CASES, ids=lambda l: l.label)
def test_edge_cases(layer):
    _full_case(layer)


def test_window_at_least_T_equals_causal():
    """A window as wide as the sequence removes nothing: bit-identical to full causal."""
    gu.require_gpu()
    a = _full_case(_layer(1, 320, 320, 4, 2, 0, seed=31))
    b = _full_case(_layer(1, 320, 320, 4, 2, 320, seed=31))
    c = _full_case(_layer(1, 320, 320, 4, 2, 100000, seed=31))
    assert torch.equal(a, b) and torch.equal(a, c)


def test_deterministic():
    gu.require_gpu()
    a = _full_case(_layer(1, 256, 256, 4, 1, 70, seed=41))
    b = _full_case(_layer(1, 256, 256, 4, 1, 70, seed=41))
    assert torch.equal(a, b)


def _sampled_case(layer: PrefillLayer, n_rows: int, seed: int):
    gu.require_gpu()
    x = prefill_inputs(layer)
    q, k, v = gu.to_cuda(x.q, x.k, x.v)
    table = gu.rope_table(layer.d, layer.rope, layer.S)
    o, lse = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S)
    rows = gu.sample_rows(layer.B, layer.Hq, layer.Hkv, layer.T, layer.window, n_rows, seed)
    w = gu.oracle_freq(layer.d, layer.rope)
    ro, rl = gu.orc().attention(x.q, x.k, x.v, window=layer.window, scale=layer.scale, w=w,
                                amp=layer.rope.amp, rows=rows)
    idx = torch.from_numpy(rows.astype(np.int64))
    og = o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = lse.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    gu.compare(og, ro, what=layer.label + " sampled")
    gu.compare(lg, rl, what=layer.label + " sampled lse")
    assert torch.isfinite(o).all()


def test_medium_window_sampled():
    _sampled_case(_layer(1, 4096, 4096, 16, 2, 2048, seed=51), 1024, 1)


def test_plamo3_local_prefill_full_size_sampled():
    """B=2, T=S=8192, 64/8 heads, d=128, W=2048 -- the benchmark's launch."""
    _sampled_case(WORKLOADS["plamo3_local_prefill"].layers[0], 4096, 2)


def test_plamo3_global_prefill_full_size_sampled():
    """B=1, T=S=32768, 64/8 heads, YaRN (s=8), logits x1.2, full causal."""
    _sampled_case(WORKLOADS["plamo3_global_prefill"].layers[0], 4096, 3)


# ---- wide heads (Gemma-4 shapes: d = 256 local, d = 512 global with partial RoPE) ----
PROPE = RopeSpec(base=1e6, rotate_fraction=0.25)

WIDE_CASES = [
    _layer(1, 200, 200, 2, 1, 0, d=256, seed=61),
    _layer(1, 130, 130, 4, 2, 1, d=256, seed=62),
    _layer(1, 300, 300, 4, 2, 64, d=256, seed=63),
    _layer(2, 257, 257, 4, 4, 127, d=256, seed=64),
    _layer(1, 100, 333, 6, 2, 0, d=256, seed=65),
    _layer(1, 200, 200, 2, 1, 0, PROPE, d=512, seed=71),
    _layer(1, 130, 130, 8, 1, 5, PROPE, d=512, seed=72),
    _layer(1, 300, 300, 4, 2, 0, PROPE, d=512, seed=73),
    _layer(1, 65, 500, 8, 2, 100, PROPE, d=512, seed=74),
    _layer(1, 1, 1, 2, 1, 0, d=512, seed=75),
    # odd groups at d = 512: the cluster's second head pair repeats the group's last head
    _layer(1, 260, 260, 3, 1, 0, PROPE, d=512, seed=76),
    _layer(1, 200, 330, 6, 2, 70, PROPE, d=512, seed=77),
    _layer(2, 129, 129, 2, 2, 0, d=512, seed=78),
]


@pytest.mark.parametrize("layer", WIDE_CASES, ids=lambda l: l.label)
def test_wide_head_edge_cases(layer):
    _full_case(layer)


@pytest.mark.parametrize("index", range(6))
def test_gemma4_period_layer_full_size_sampled(index):
    """Every layer of the Gemma-4-shaped period at full size (T=S=16384, 16 query heads):
    layers 0-4 d=256, 8 KV heads, window 1024; layer 5 d=512, 2 KV heads, full causal,
    partial RoPE.  4096 sampled rows per layer, covering every head of two KV groups and
    the window, tile and sequence edges."""
    _sampled_case(WORKLOADS["gemma4_period_6layer"].layers[index], 4096, 40 + index)


@pytest.mark.parametrize("name,index", [("plamo3_local_prefill", 0),
                                        ("gemma4_period_6layer", 0),
                                        ("gemma4_period_6layer", 5)])
def test_full_size_repeat_bitwise(name, index):
    """Full-size launches repeated back to back give bit-identical outputs: a result that
    depended on the timing of the asynchronous pipeline (a barrier phase observed too
    early, a buffer overwritten while still being read) would show up as a difference."""
    gu.require_gpu()
    layer = WORKLOADS[name].layers[index]
    x = prefill_inputs(layer)
    q, k, v = gu.to_cuda(x.q, x.k, x.v)
    table = gu.rope_table(layer.d, layer.rope, layer.S)
    first, first_lse = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S)
    for _ in range(6):
        o, lse = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S)
        assert torch.equal(o, first) and torch.equal(lse, first_lse)


def test_persistent_odd_group_many_items_sampled():
    """Windowed layer with more items than SMs (each persistent CTA walks several) and an
    odd group size, so single-tile items alternate with two-tile ones."""
    layer = _layer(1, 8192, 8192, 12, 4, 256, seed=81)
    from global_causal_gqa_gb300 import accounting as acc
    assert acc.prefill_d128_kernel(layer.T, layer.S, layer.window) == "prefill_persistent_kernel"
    _sampled_case(layer, 2048, 6)


def test_stream_kernel_medium_causal_sampled():
    """Causal sweep long enough (mean >= 48 key tiles per query block) for the
    one-CTA-per-item kernel, with a ragged last block and queries after a longer history."""
    layer = _layer(1, 12200, 12300, 4, 2, 0, YARN, seed=82)
    from global_causal_gqa_gb300 import accounting as acc
    assert acc.prefill_d128_kernel(layer.T, layer.S, layer.window) == "prefill_kernel"
    _sampled_case(layer, 2048, 7)


def test_wide_many_items_sampled():
    """d = 256 windowed layer with far more query blocks than SMs, a history before the
    queries, ragged windows and single-tile query blocks."""
    _sampled_case(_layer(2, 4000, 4100, 8, 4, 384, d=256, seed=83), 2048, 8)


def test_wide_single_tile_items():
    """Every query block a single key tile (window 1 at d = 256)."""
    _full_case(_layer(1, 1100, 1100, 4, 2, 1, d=256, seed=84))


def test_wide_long_causal_sampled():
    """d = 256 causal sweep over 97 query blocks of up to 97 key tiles each."""
    _sampled_case(_layer(1, 12400, 12400, 2, 1, 0, d=256, seed=85), 1024, 9)


# ---- RoPE on K fused into the tile load (k_is_rotated = 2, d = 128) ----
FUSED_CASES = [
    _layer(1, 200, 200, 2, 1, 0, seed=91),
    _layer(1, 300, 300, 4, 1, 4, seed=92),
    _layer(1, 384, 384, 2, 1, 129, seed=93),
    _layer(2, 257, 257, 6, 2, 64, YARN, seed=94),
    _layer(1, 160, 160, 3, 1, 0, seed=95),
    _layer(1, 129, 700, 4, 2, 200, YARN, seed=96),
    _layer(1, 2000, 2000, 16, 2, 0, seed=97),   # long causal items: still the fused kernel
]


@pytest.mark.parametrize("layer", FUSED_CASES, ids=lambda l: l.label)
def test_fused_k_rope_equals_rotate_once(layer):
    """K's rotation fused into the tile load gives the rotate-once result bit for bit (the
    same fp32 rotation of the same bf16 keys, rounded once), and matches the oracle."""
    gu.require_gpu()
    x = prefill_inputs(layer)
    q, k, v = gu.to_cuda(x.q, x.k, x.v)
    table = gu.rope_table(layer.d, layer.rope, layer.S)
    o0, l0 = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S, k_mode=0)
    o2, l2 = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S, k_mode=2)
    assert torch.equal(o0, o2) and torch.equal(l0, l2)
    w = gu.oracle_freq(layer.d, layer.rope)
    ro, rl = gu.orc().attention(x.q, x.k, x.v, window=layer.window, scale=layer.scale, w=w,
                                amp=layer.rope.amp)
    gu.compare(o2, ro, what=layer.label + " fused K")
    gu.compare(l2, rl, what=layer.label + " fused K lse")


def test_fused_k_rope_full_size_local_layer():
    """The PLaMo-3-shaped local layer (B=2, T=S=8192, 64/8 heads, W=2048) with the fused
    form: equal to the rotate-once result bit for bit."""
    gu.require_gpu()
    layer = WORKLOADS["plamo3_local_prefill"].layers[0]
    x = prefill_inputs(layer)
    q, k, v = gu.to_cuda(x.q, x.k, x.v)
    table = gu.rope_table(layer.d, layer.rope, layer.S)
    o0, l0 = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S, k_mode=0)
    o2, l2 = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S, k_mode=2)
    assert torch.equal(o0, o2) and torch.equal(l0, l2)
