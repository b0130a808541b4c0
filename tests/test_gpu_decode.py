"""Decode-step parity: gqa_kv_append + gqa_attn_decode (C-ABI) against the oracle.

Slots written and the updated counts must match the oracle's cache index model
bit-exactly; outputs within max abs 2e-2 / mean abs 2e-3 of the fp64 oracle.
"""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from workloads import WORKLOADS, RopeSpec, decode_inputs
from workloads.gen import DecodeInputs

pytestmark = pytest.mark.gpu

LOCAL = RopeSpec(base=1e4)
YARN = RopeSpec(base=1e6, yarn_factor=8.0, amp=math.sqrt(1.2))


class DecodeSetup:
    """Device copies of one decode batch plus its descriptor array."""

    def __init__(self, x: DecodeInputs, d: int, slack: int = 4):
        self.x = x
        self.d = d
        self.q = x.q.cuda()
        self.k_new = x.k_new.cuda()
        self.v_new = x.v_new.cuda()
        self.kc = [t.cuda() for t in x.k_cache]
        self.vc = [t.cuda() for t in x.v_cache]
        # one table per distinct RoPE setting, long enough for every sequence using it
        self.tables = {}
        for i, r in enumerate(x.rope):
            need = x.cap[i] if x.is_ring[i] else x.count_before[i] + 1 + slack
            cur = self.tables.get(r, (None, 0))[1]
            self.tables[r] = (None, max(cur, need))
        for r, (_, n) in list(self.tables.items()):
            self.tables[r] = (gu.rope_table(d, r, n), n)
        a = gqa.make_kv_descs(self.kc, self.vc, [self.tables[r][0] for r in x.rope], x.cap,
                              x.count_before, x.is_ring, [self.tables[r][1] for r in x.rope])
        self.desc_host = a
        self.descs = torch.from_numpy(a.view(np.uint8).copy()).cuda()

    def counts(self):
        a = self.descs.cpu().numpy().view(gqa.KV_DESC_DTYPE)
        return a["count"].astype(np.int64)


def run_step(st: DecodeSetup, Hq: int, Hkv: int, scale: float, max_len: int):
    nseq = st.q.shape[0]
    slots = torch.full((nseq,), -7, dtype=torch.int32, device="cuda")
    gqa.gqa_kv_append(st.descs, nseq, st.k_new, st.v_new, Hkv, st.d, slots)
    o = torch.empty_like(st.q)
    lse = torch.empty(nseq, Hq, dtype=torch.float32, device="cuda")
    wsb = gqa.gqa_decode_workspace_bytes(nseq, Hq, Hkv, st.d, max_len)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    gqa.gqa_attn_decode(st.q, st.descs, nseq, Hq, Hkv, st.d, scale, max_len, o, lse, ws, wsb)
    status = gqa.gqa_get_device_status()
    assert status == 0, gqa.STATUS_NAMES.get(status, status)
    return o, lse, slots


def oracle_step(x: DecodeInputs, d: int, scale: float):
    w = [gu.oracle_freq(d, r) for r in x.rope]
    amp = [r.amp for r in x.rope]
    return gu.orc().decode_step(x.q, x.k_new, x.v_new, x.k_cache, x.v_cache, x.cap,
                                x.count_before, x.is_ring, w, amp, scale)


def _random_batch(lengths, rings, Hq, Hkv, d=128, seed=0):
    """lengths: for linear caches the count before the append; rings: (cap, n_before)."""
    g = torch.Generator().manual_seed(seed)
    nseq = len(lengths) + len(rings)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    q, kn, vn = bf(nseq, Hq, d), bf(nseq, Hkv, d), bf(nseq, Hkv, d)
    kc, vc, cap, cnt, ring, rope = [], [], [], [], [], []
    for n in lengths:
        c = n + 1 + int(torch.randint(0, 3, (1,), generator=g))
        kc.append(bf(Hkv, c, d)); vc.append(bf(Hkv, c, d))
        cap.append(c); cnt.append(n); ring.append(0); rope.append(YARN)
    for c, n in rings:
        kc.append(bf(Hkv, c, d)); vc.append(bf(Hkv, c, d))
        cap.append(c); cnt.append(n); ring.append(1); rope.append(LOCAL)
    return DecodeInputs(q, kn, vn, kc, vc, cap, cnt, ring, rope)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (64, 8), (16, 8), (6, 2)])
def test_mixed_small_batch(Hq, Hkv):
    """Linear caches across split and block boundaries; rings before, at and after
    wrap-around, including a ring that is not full yet."""
    gu.require_gpu()
    lengths = [0, 14, 15, 16, 17, 1023, 1024, 1025, 2500]
    rings = [(64, 0), (64, 10), (64, 63), (64, 64), (64, 200), (2048, 2047), (2048, 5000),
             (100, 349)]
    x = _random_batch(lengths, rings, Hq, Hkv, seed=Hq * 7 + Hkv)
    st = DecodeSetup(x, 128)
    scale = 1 / math.sqrt(128)
    o, lse, slots = run_step(st, Hq, Hkv, scale, max_len=4096)
    ro, rl, rslots, rcounts = oracle_step(x, 128, scale)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), rslots)
    assert np.array_equal(st.counts(), rcounts)
    gu.compare(o, ro, what=f"decode Hq={Hq} Hkv={Hkv}")
    gu.compare(lse, rl, what="decode lse")


def test_cache_rows_written_exactly():
    gu.require_gpu()
    x = _random_batch([5, 9], [(8, 13)], 4, 2, seed=3)
    st = DecodeSetup(x, 128)
    run_step(st, 4, 2, 0.1, max_len=64)
    for i, slot in enumerate([5, 9, 13 % 8]):
        assert torch.equal(st.kc[i][:, slot].cpu(), x.k_new[i])
        assert torch.equal(st.vc[i][:, slot].cpu(), x.v_new[i])
        # every other slot untouched
        keep = [s for s in range(x.cap[i]) if s != slot]
        assert torch.equal(st.kc[i][:, keep].cpu(), x.k_cache[i][:, keep])


def test_two_steps_in_a_row():
    """Two append+decode steps: the second sees the first step's token."""
    gu.require_gpu()
    x = _random_batch([30, 1030], [(64, 70)], 8, 2, seed=5)
    for c in range(2):
        x.cap[c] += 2
        x.k_cache[c] = torch.cat([x.k_cache[c], torch.zeros(2, 2, 128, dtype=torch.bfloat16)], 1)
        x.v_cache[c] = torch.cat([x.v_cache[c], torch.zeros(2, 2, 128, dtype=torch.bfloat16)], 1)
    st = DecodeSetup(x, 128)
    run_step(st, 8, 2, 0.1, max_len=2048)
    # the oracle's second step starts from the caches as the GPU left them
    x2 = replace(x, k_cache=[t.cpu() for t in st.kc], v_cache=[t.cpu() for t in st.vc],
                 count_before=[int(c) for c in st.counts()])
    o, _, _ = run_step(st, 8, 2, 0.1, max_len=2048)
    ro, _, _, _ = oracle_step(x2, 128, 0.1)
    gu.compare(o, ro, what="second step")


def test_full_linear_cache_reports_capacity():
    gu.require_gpu()
    x = _random_batch([4], [], 2, 1, seed=9)
    x.cap[0] = 4
    x.k_cache[0] = x.k_cache[0][:, :4].contiguous()
    x.v_cache[0] = x.v_cache[0][:, :4].contiguous()
    st = DecodeSetup(x, 128)
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    gqa.gqa_kv_append(st.descs, 1, st.k_new, st.v_new, 1, 128, slots)
    assert gqa.gqa_get_device_status() == -4
    assert slots.item() == -1 and st.counts()[0] == 4
    assert gqa.gqa_get_device_status() == 0  # cleared by the read


def test_plamo3_decode_batch_full_size():
    """32 sequences: 16 global caches S ~ U{8192..65536} (YaRN s=8, logits x1.2) and 16
    local rings of 2048 -- the benchmark's workload, every output compared."""
    gu.require_gpu()
    w = WORKLOADS["plamo3_decode_batch32"]
    x = decode_inputs(w)
    st = DecodeSetup(x, w.d)
    max_len = max(w.global_len_range[1], w.window)
    o, lse, slots = run_step(st, w.Hq, w.Hkv, w.scale, max_len)
    ro, rl, rslots, rcounts = oracle_step(x, w.d, w.scale)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), rslots)
    assert np.array_equal(st.counts(), rcounts)
    gu.compare(o, ro, what="plamo3 decode")
    gu.compare(lse, rl, what="plamo3 decode lse")


PROPE = RopeSpec(base=1e6, rotate_fraction=0.25)


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 8, 256), (16, 2, 512), (8, 1, 256), (32, 4, 512),
                                      (6, 3, 256)])
def test_wide_head_decode(Hq, Hkv, d):
    """Gemma-4 head dims: d = 256 (local layers) and 512 (global), streamed by 2 or 4 warps
    per KV head; linear caches across split boundaries and rings around wrap-around."""
    gu.require_gpu()
    lengths = [0, 15, 1023, 1024, 2100]
    rings = [(64, 10), (64, 200), (1024, 1023), (1024, 3000)]
    x = _random_batch(lengths, rings, Hq, Hkv, d, seed=Hq + Hkv + d)
    if d == 512:
        x = replace(x, rope=[PROPE if not r else LOCAL for r in x.is_ring])
    st = DecodeSetup(x, d)
    scale = 1 / math.sqrt(d)
    o, lse, slots = run_step(st, Hq, Hkv, scale, max_len=4096)
    ro, rl, rslots, rcounts = oracle_step(x, d, scale)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), rslots)
    assert np.array_equal(st.counts(), rcounts)
    gu.compare(o, ro, what=f"decode d={d} Hq={Hq} Hkv={Hkv}")
    gu.compare(lse, rl, what="decode lse")


def test_prope_unrotated_parts_match_rotation():
    """d = 512 with p-RoPE: a part whose 64 pairs never rotate (table rows 0 and 1 both
    (1, 0)) skips the table rows and the rotation.  Forcing the rotation on those parts --
    row 1 of pairs 64..255 given sin = 1e-30, which leaves every bf16 key of a normal
    sample as it is -- gives the same output and lse bit for bit."""
    gu.require_gpu()
    Hq, Hkv, d = 16, 2, 512
    x = _random_batch([5, 700, 2100], [], Hq, Hkv, d, seed=4242)
    x = replace(x, rope=[PROPE] * 3)
    st = DecodeSetup(x, d)
    scale = 1 / math.sqrt(d)
    o1, lse1, _ = run_step(st, Hq, Hkv, scale, max_len=4096)
    tab, n = st.tables[PROPE]
    t2 = tab.clone().view(n, d // 2, 2)
    t2[1, 64:, 1] = 1e-30
    t2 = t2.view(-1)
    a = gqa.make_kv_descs(st.kc, st.vc, [t2] * 3, x.cap, st.counts().tolist(), x.is_ring,
                          [n] * 3)
    descs2 = torch.from_numpy(a.view(np.uint8).copy()).cuda()
    o2 = torch.empty_like(st.q)
    lse2 = torch.empty_like(lse1)
    wsb = gqa.gqa_decode_workspace_bytes(3, Hq, Hkv, d, 4096)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    gqa.gqa_attn_decode(st.q, descs2, 3, Hq, Hkv, d, scale, 4096, o2, lse2, ws, wsb)
    assert gqa.gqa_get_device_status() == 0
    assert torch.equal(o1, o2)
    assert torch.equal(lse1, lse2)


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (32, 32)])
def test_long_split_boundaries(Hq, Hkv):
    """max_len 8192: caches ending just before, at and after split boundaries, a split
    that holds a single key, and rings that wrap.  With 2 KV heads the batch gets 512-key
    splits; with 32 (four CTAs of 8 heads per sequence) the longest, 2048-key splits."""
    gu.require_gpu()
    lengths = [2047, 2048, 2049, 4095, 4096, 4097, 6143]
    rings = [(2048, 2047), (2048, 5000)]
    x = _random_batch(lengths, rings, Hq, Hkv, seed=77)
    st = DecodeSetup(x, 128)
    scale = 1 / math.sqrt(128)
    o, lse, slots = run_step(st, Hq, Hkv, scale, max_len=8192)
    ro, rl, rslots, rcounts = oracle_step(x, 128, scale)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), rslots)
    assert np.array_equal(st.counts(), rcounts)
    gu.compare(o, ro, what=f"decode, long splits, Hkv={Hkv}")
    gu.compare(lse, rl, what=f"decode lse, long splits, Hkv={Hkv}")


@pytest.mark.parametrize("nseq_lin,Hq,Hkv,d,max_len",
                         [(1, 1, 1, 128, 64), (3, 3, 1, 128, 320), (1, 5, 1, 256, 192),
                          (3, 7, 1, 128, 448), (1, 3, 1, 512, 320), (3, 1, 1, 128, 6208)])
def test_odd_partial_counts(nseq_lin, Hq, Hkv, d, max_len):
    """nseq * Hq * nsplit odd: the (m, l) pairs of the workspace fill an odd number of
    8-byte slots, and the O partials after them must still start on a 16-byte boundary
    (they are written with 16-byte stores).  The split count is read back from the
    workspace size (whole partials of d + 2 floats per sequence, head and split)."""
    gu.require_gpu()
    lengths = [max_len - 1 - 97 * i for i in range(nseq_lin - 1)] + [min(40, max_len - 1)]
    x = _random_batch(lengths, [], Hq, Hkv, d, seed=1000 + Hq * 10 + nseq_lin)
    if d == 512:
        x = replace(x, rope=[PROPE] * len(lengths))
    nseq = len(lengths)
    wsb = gqa.gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len)
    nsplit = (wsb // 4) // (nseq * Hq * (d + 2))
    assert (nseq * Hq * nsplit) % 2 == 1, nsplit
    st = DecodeSetup(x, d)
    scale = 1 / math.sqrt(d)
    o, lse, slots = run_step(st, Hq, Hkv, scale, max_len=max_len)
    ro, rl, rslots, rcounts = oracle_step(x, d, scale)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), rslots)
    assert np.array_equal(st.counts(), rcounts)
    gu.compare(o, ro, what=f"decode nseq={nseq} Hq={Hq} d={d} max_len={max_len}")
    gu.compare(lse, rl, what="decode lse")


@pytest.mark.parametrize("name", ["gemma4_decode_global", "gemma4_decode_local"])
def test_gemma4_decode_batch_full_size(name):
    """The benchmark's Gemma-4-shaped decode batches in the launch the benchmark times:
    32 linear caches of 8192..65536 tokens at d = 512 (2 KV heads, p-RoPE), and 32 rings
    of 1024 at d = 256 (8 KV heads).  Every slot and count is checked bit for bit; the
    outputs of every ring, and of the longest, the shortest and 4 seeded linear caches,
    are compared with the oracle."""
    gu.require_gpu()
    w = WORKLOADS[name]
    x = decode_inputs(w)
    st = DecodeSetup(x, w.d)
    max_len = max(w.global_len_range[1], w.window)
    o, lse, slots = run_step(st, w.Hq, w.Hkv, w.scale, max_len)
    orc = gu.orc()
    want_slots = [orc.append_slot(r, c, cap) for r, c, cap in zip(x.is_ring, x.count_before,
                                                                    x.cap)]
    assert slots.cpu().tolist() == want_slots
    assert st.counts().tolist() == [c + 1 for c in x.count_before]
    if w.n_global:
        lens = np.array(x.count_before)
        rng = np.random.default_rng(12)
        idx = sorted({int(lens.argmax()), int(lens.argmin())} |
                     set(rng.choice(w.nseq, 4, replace=False).tolist()))
    else:
        idx = list(range(w.nseq))
    sub = lambda a: [a[i] for i in idx]  # noqa: E731
    xs = DecodeInputs(x.q[idx], x.k_new[idx], x.v_new[idx], sub(x.k_cache), sub(x.v_cache),
                      sub(x.cap), sub(x.count_before), sub(x.is_ring), sub(x.rope))
    ro, rl, rslots, _ = oracle_step(xs, w.d, w.scale)
    assert rslots.tolist() == [want_slots[i] for i in idx]
    gu.compare(o[idx], ro, what=f"{name} ({len(idx)} sequences)")
    gu.compare(lse[idx], rl, what=f"{name} lse")
