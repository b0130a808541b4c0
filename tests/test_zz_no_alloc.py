"""gqa_attn_decode_static: decode for callers that cannot allocate device memory.

Such callers (a host whose GPU memory is owned by another allocator, a serving loop that
must not allocate per step) call this entry point without a workspace; the library keeps
the split-KV partials in a fixed 16 MiB device array of its own.  These tests call it
through the C ABI and check it against gqa_attn_decode (caller-provided workspace) on two
calls in a row, at the tolerance the other decode tests use, and check the size limit.
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


def _batch(seed, Hq=64, Hkv=8, d=128):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    lin = [3, 1000, 1024, 2049, 4000]            # tokens held before the append
    rings = [(2048, 2047), (2048, 9000), (64, 70)]
    n = len(lin) + len(rings)
    kc, vc, cap, cnt, ring, rope = [], [], [], [], [], []
    for c in lin:
        kc.append(bf(Hkv, c + 2, d)); vc.append(bf(Hkv, c + 2, d))
        cap.append(c + 2); cnt.append(c); ring.append(0)
        rope.append(RopeSpec(base=1e6, yarn_factor=8.0, amp=math.sqrt(1.2)))
    for c, k in rings:
        kc.append(bf(Hkv, c, d)); vc.append(bf(Hkv, c, d))
        cap.append(c); cnt.append(k); ring.append(1); rope.append(RopeSpec(base=1e4))
    return DecodeInputs(bf(n, Hq, d), bf(n, Hkv, d), bf(n, Hkv, d), kc, vc, cap, cnt, ring,
                        rope)


class _Dev:
    def __init__(self, x, d=128):
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
        self.descs0 = torch.from_numpy(a.view(np.uint8).copy()).cuda()
        self.descs = self.descs0.clone()
        self.n = len(x.cap)
        # the appended token is written once; both paths then read the same caches
        gqa.gqa_kv_append(self.descs, self.n, self.kn, self.vn, self.kn.shape[1], d)


def _reference(dev, Hq, Hkv, max_len, scale):
    o = torch.empty_like(dev.q)
    lse = torch.empty(dev.n, Hq, dtype=torch.float32, device="cuda")
    wsb = gqa.gqa_decode_workspace_bytes(dev.n, Hq, 128, max_len)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    gqa.gqa_attn_decode(dev.q, dev.descs, dev.n, Hq, Hkv, 128, scale, max_len, o, lse, ws, wsb)
    assert gqa.gqa_get_device_status() == 0
    return o, lse


def _static(dev, Hq, Hkv, max_len, scale):
    o = torch.full_like(dev.q, float("nan"))
    lse = torch.full((dev.n, Hq), float("nan"), dtype=torch.float32, device="cuda")
    gqa.gqa_attn_decode_static(dev.q, dev.descs, dev.n, Hq, Hkv, 128, scale, max_len, o, lse)
    assert gqa.gqa_get_device_status() == 0
    return o, lse


def test_static_matches_workspace_decode_twice():
    gu.require_gpu()
    Hq, Hkv, max_len, scale = 64, 8, 4096, 1 / math.sqrt(128)
    assert gqa.gqa_decode_workspace_bytes(8, Hq, 128, max_len) <= STATIC_BYTES
    dev_a = _Dev(_batch(1))
    dev_b = _Dev(_batch(2))
    ref_a, lref_a = _reference(dev_a, Hq, Hkv, max_len, scale)
    ref_b, lref_b = _reference(dev_b, Hq, Hkv, max_len, scale)
    # two calls in a row on different inputs: the second must not see the first's partials
    o1, l1 = _static(dev_a, Hq, Hkv, max_len, scale)
    o2, l2 = _static(dev_b, Hq, Hkv, max_len, scale)
    for o, r, l, lr in ((o1, ref_a, l1, lref_a), (o2, ref_b, l2, lref_b)):
        assert torch.isfinite(o.float()).all() and torch.isfinite(l).all()
        gu.compare(o, r.float().cpu().numpy().astype(np.float64), what="static vs workspace")
        gu.compare(l, lr.cpu().numpy().astype(np.float64), what="static lse")


def test_static_rejects_oversize_without_launch():
    gu.require_gpu()
    Hq, Hkv = 64, 8
    dev = _Dev(_batch(3))
    max_len = 1 << 20                      # partials far beyond the 16 MiB array
    assert gqa.gqa_decode_workspace_bytes(dev.n, Hq, 128, max_len) > STATIC_BYTES
    o = torch.zeros_like(dev.q)
    st = gqa.gqa_attn_decode_static(dev.q, dev.descs, dev.n, Hq, Hkv, 128, 0.1, max_len, o,
                                    None, check=False)
    assert gqa.STATUS_NAMES[st] == "GQA_ERR_WORKSPACE"
    assert gqa.gqa_get_device_status() == 0
    assert torch.count_nonzero(o).item() == 0
