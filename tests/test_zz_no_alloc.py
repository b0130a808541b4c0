"""gqa_attn_decode_static: decode for callers that cannot allocate device memory.

Such callers (a host whose GPU memory is owned by another allocator, a serving loop that
must not allocate per step) call this entry point without a workspace; the library keeps
the split-KV partials in a fixed 16 MiB device array of its own.  These tests call it
through the C ABI and check it against gqa_attn_decode (caller-provided workspace) on two
calls in a row: the same kernels run, so output and lse must be equal bit for bit.  The
two calls differ in batch size, head count and split layout, so the second one would read
stale partials of the first if the array were not rewritten where it is read.  The first
call is also compared with the fp64 oracle at the tolerance of the other decode tests.
The file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from workloads import RopeSpec
from workloads.gen import DecodeInputs

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20
GLOBAL = RopeSpec(base=1e6, yarn_factor=8.0, amp=math.sqrt(1.2))
LOCAL = RopeSpec(base=1e4)


def _batch(seed, lin, rings, Hq, Hkv, d=128):
    """lin: tokens held before the append (linear caches); rings: (cap, tokens appended)."""
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    n = len(lin) + len(rings)
    kc, vc, cap, cnt, ring, rope = [], [], [], [], [], []
    for c in lin:
        kc.append(bf(Hkv, c + 2, d)); vc.append(bf(Hkv, c + 2, d))
        cap.append(c + 2); cnt.append(c); ring.append(0); rope.append(GLOBAL)
    for c, k in rings:
        kc.append(bf(Hkv, c, d)); vc.append(bf(Hkv, c, d))
        cap.append(c); cnt.append(k); ring.append(1); rope.append(LOCAL)
    return DecodeInputs(bf(n, Hq, d), bf(n, Hkv, d), bf(n, Hkv, d), kc, vc, cap, cnt, ring,
                        rope)


class _Dev:
    def __init__(self, x, d=128):
        self.x = x
        self.q, self.kn, self.vn = x.q.cuda(), x.k_new.cuda(), x.v_new.cuda()
        self.kc = [t.cuda() for t in x.k_cache]
        self.vc = [t.cuda() for t in x.v_cache]
        tables = {}
        for r in set(x.rope):
            n = max(x.cap[i] for i in range(len(x.cap)) if x.rope[i] == r)
            tables[r] = (gu.rope_table(d, r, n), n)
        self.tables = tables
        a = gqa.make_kv_descs(self.kc, self.vc, [tables[r][0] for r in x.rope], x.cap,
                              x.count_before, x.is_ring, [tables[r][1] for r in x.rope])
        self.descs = torch.from_numpy(a.view(np.uint8).copy()).cuda()
        self.n = len(x.cap)
        # the appended token is written once; both paths then read the same caches
        gqa.gqa_kv_append(self.descs, self.n, self.kn, self.vn, self.kn.shape[1], d)


def _workspace_decode(dev, Hq, Hkv, max_len, scale):
    o = torch.empty_like(dev.q)
    lse = torch.empty(dev.n, Hq, dtype=torch.float32, device="cuda")
    wsb = gqa.gqa_decode_workspace_bytes(dev.n, Hq, Hkv, 128, max_len)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    gqa.gqa_attn_decode(dev.q, dev.descs, dev.n, Hq, Hkv, 128, scale, max_len, o, lse, ws, wsb)
    assert gqa.gqa_get_device_status() == 0
    return o, lse


def _static_decode(dev, Hq, Hkv, max_len, scale):
    o = torch.full_like(dev.q, float("nan"))
    lse = torch.full((dev.n, Hq), float("nan"), dtype=torch.float32, device="cuda")
    gqa.gqa_attn_decode_static(dev.q, dev.descs, dev.n, Hq, Hkv, 128, scale, max_len, o, lse)
    assert gqa.gqa_get_device_status() == 0
    return o, lse


def test_static_matches_workspace_decode_twice():
    gu.require_gpu()
    scale = 1 / math.sqrt(128)
    # call A: 8 sequences, 64/8 heads, max_len 8192
    a_shape = dict(Hq=64, Hkv=8, max_len=8192)
    dev_a = _Dev(_batch(1, [3, 1000, 2049, 4000, 8000], [(2048, 2047), (2048, 9000), (64, 70)],
                        a_shape["Hq"], a_shape["Hkv"]))
    # call B: 3 sequences, 3/1 heads, max_len 704: another split layout, so every record
    # sits at another offset than in call A, and nseq * Hq * nsplit is odd
    b_shape = dict(Hq=3, Hkv=1, max_len=704)
    dev_b = _Dev(_batch(2, [700, 5], [(256, 300)], b_shape["Hq"], b_shape["Hkv"]))
    splits = []
    for dev, shp in ((dev_a, a_shape), (dev_b, b_shape)):
        wsb = gqa.gqa_decode_workspace_bytes(dev.n, shp["Hq"], shp["Hkv"], 128, shp["max_len"])
        assert wsb <= STATIC_BYTES
        splits.append((wsb // 4) // (dev.n * shp["Hq"] * 130))
    assert splits[0] != splits[1] and (dev_b.n * b_shape["Hq"] * splits[1]) % 2 == 1
    ref_a = _workspace_decode(dev_a, scale=scale, **a_shape)
    ref_b = _workspace_decode(dev_b, scale=scale, **b_shape)
    # two calls in a row; the second must read none of the first's partials
    got_a = _static_decode(dev_a, scale=scale, **a_shape)
    got_b = _static_decode(dev_b, scale=scale, **b_shape)
    for got, ref, name in ((got_a, ref_a, "A"), (got_b, ref_b, "B")):
        assert torch.equal(got[0], ref[0]), f"call {name}: output differs from gqa_attn_decode"
        assert torch.equal(got[1], ref[1]), f"call {name}: lse differs from gqa_attn_decode"
    # and the first call against the fp64 oracle
    x = dev_a.x
    w = [gu.oracle_freq(128, r) for r in x.rope]
    ro, rl, _, _ = gu.orc().decode_step(x.q, x.k_new, x.v_new, x.k_cache, x.v_cache, x.cap,
                                        x.count_before, x.is_ring, w, [r.amp for r in x.rope],
                                        scale)
    gu.compare(got_a[0], ro, what="static decode vs oracle")
    gu.compare(got_a[1], rl, what="static decode lse vs oracle")


def test_static_rejects_oversize_without_launch():
    gu.require_gpu()
    Hq, Hkv = 64, 8
    dev = _Dev(_batch(3, [3, 1000], [(64, 70)], Hq, Hkv))
    max_len = 1 << 20                      # partials far beyond the 16 MiB array
    assert gqa.gqa_decode_workspace_bytes(dev.n, Hq, Hkv, 128, max_len) > STATIC_BYTES
    o = torch.zeros_like(dev.q)
    st = gqa.gqa_attn_decode_static(dev.q, dev.descs, dev.n, Hq, Hkv, 128, 0.1, max_len, o,
                                    None, check=False)
    assert gqa.STATUS_NAMES[st] == "GQA_ERR_WORKSPACE"
    assert gqa.gqa_get_device_status() == 0
    assert torch.count_nonzero(o).item() == 0
