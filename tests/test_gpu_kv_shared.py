"""Shared K/V projection (Gemma 4 global layers, attention_k_eq_v) against the fp64 oracle.

One projection output Z per token gives both K = RoPE(N_{gamma_k}(Z)) and V = N_1(Z)
("PLaMo 3アーキテクチャ徹底解析" §5.2 and the Gemma 4 comparison of §8); the query is
N_{gamma_q}(q), rotated.  The library caches only Zn = N_1(Z) and recomputes the keys.
Prefill: gqa_qk_norm_rope_kv_shared, then gqa_attn_prefill over (k_rot, v_out).  Decode:
caches of Zn made from raw Z rows by the same norm pass, then gqa_kv_shared_append and
gqa_attn_decode_kv_shared.  The oracle computes every norm from the raw bf16 rows in
fp64.  Scale 1 (Gemma), with gains that give logits of standard deviation ~1.

The bar is the one every attention test uses, max abs 2e-2 / mean abs 2e-3 on the bf16
outputs, end to end: from the raw rows, against the definition computed in fp64 with no
bf16 storage anywhere.  The measured errors are printed.  Slots and counts bit-exact.
"""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from test_gpu_decode import LOCAL, YARN, DecodeSetup, _random_batch
from workloads import RopeSpec, decode_inputs, get_workload, norm_gains

pytestmark = pytest.mark.gpu

EPS = 1e-6
PROPE = RopeSpec(base=1e6, rotate_fraction=0.25)


def _bf(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _dev_gain(g: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(g).to(torch.float32).cuda()


def _report(gpu, ref, what):
    mx, mn = gu.compare(gpu, ref, what=what)
    print(f"{what}: max abs {mx:.3e}, mean abs {mn:.3e}")


@pytest.mark.parametrize("d,Hq,Hkv,T,window,rope", [
    (512, 8, 2, 300, 0, PROPE),
    (256, 8, 4, 333, 128, LOCAL),
    (128, 8, 2, 260, 0, YARN),
    (128, 6, 3, 200, 64, LOCAL),
])
def test_prefill_kv_shared(d, Hq, Hkv, T, window, rope):
    gu.require_gpu()
    B = 1
    q = _bf((B, Hq, T, d), 1300 + d + T)
    z = _bf((B, Hkv, T, d), 1400 + d + T, scale=3.0)     # any scale: the norms remove it
    gq, gk = norm_gains(d, 1500 + d), norm_gains(d, 1600 + d)
    table = gu.rope_table(d, rope, T)
    qd, zd = q.cuda(), z.cuda()
    q_out, v_out, k_rot = torch.empty_like(qd), torch.empty_like(zd), torch.empty_like(zd)
    gqa.gqa_qk_norm_rope_kv_shared(qd, zd, q_out, v_out, k_rot, B, Hq, Hkv, T, d, 0,
                                   _dev_gain(gq), _dev_gain(gk), EPS, table, T)
    assert gqa.gqa_get_device_status() == 0
    orc = gu.orc()
    w = gu.oracle_freq(d, rope)
    # the pass's own outputs: the values (and cache rows) Zn, the rotated keys
    gu.compare(q_out, orc.rms_norm(q, gq, EPS), what="q_out")
    gu.compare(v_out, orc.rms_norm(z, None, EPS), what="v_out = Zn")
    rk = orc.rms_norm(z, gk, EPS)
    rrot = np.stack([[[orc.rope_rotate(rk[b, h, t], t, w, rope.amp) for t in range(T)]
                      for h in range(Hkv)] for b in range(B)])
    gu.compare(k_rot, rrot, what="k_rot")
    # attention over them
    o = torch.empty_like(qd)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device="cuda")
    gqa.gqa_attn_prefill(q_out, k_rot, v_out, o, lse, B, T, T, Hq, Hkv, d, window, 1.0, table,
                         T, 1, None, 0)
    assert gqa.gqa_get_device_status() == 0
    ro, rl = orc.attention_kv_shared(q, z, q_gamma=gq, k_gamma=gk, eps=EPS, window=window,
                                     scale=1.0, w=w, amp=rope.amp)
    _report(o, ro, f"kv-shared prefill d={d} Hq={Hq} Hkv={Hkv} (end to end)")
    _report(lse, rl, f"kv-shared prefill d={d} lse (end to end)")


def _shared_setup(x, d):
    """Device caches of Zn made from the raw Z caches (x.k_cache) by the norm pass, in
    place; x.v_cache stays as a decoy the shared kernels must not read."""
    st = DecodeSetup(x, d)
    Hkv = x.k_new.shape[1]
    for i, zc in enumerate(st.kc):
        gqa.gqa_qk_norm_rope_kv_shared(None, zc, None, zc, None, 1, 0, Hkv, x.cap[i], d, 0, None,
                                       None, EPS, None, 0)
    assert gqa.gqa_get_device_status() == 0
    return st


def _shared_step(st, x, Hq, Hkv, d, gq, gk, max_len, scale=1.0):
    nseq = x.q.shape[0]
    q_out = torch.empty_like(st.q)
    slots = torch.full((nseq,), -7, dtype=torch.int32, device="cuda")
    gqa.gqa_kv_shared_append(st.descs, nseq, st.q, st.k_new, Hq, Hkv, d, _dev_gain(gq), EPS,
                             q_out, slots)
    o = torch.empty_like(st.q)
    lse = torch.empty(nseq, Hq, dtype=torch.float32, device="cuda")
    wsb = gqa.gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    gqa.gqa_attn_decode_kv_shared(q_out, st.descs, nseq, Hq, Hkv, d, scale, _dev_gain(gk),
                                  max_len, o, lse, ws, wsb)
    status = gqa.gqa_get_device_status()
    assert status == 0, gqa.STATUS_NAMES.get(status, status)
    return o, lse, slots


def _oracle_shared(x, d, gq, gk, idx=None, scale=1.0):
    """The oracle decode step over sequences idx, end to end: the definition from the raw
    rows, every norm in fp64."""
    idx = list(range(x.q.shape[0])) if idx is None else idx
    sub = lambda a: [a[i] for i in idx]  # noqa: E731
    w = [gu.oracle_freq(d, r) for r in sub(x.rope)]
    amp = [r.amp for r in sub(x.rope)]
    return gu.orc().decode_step_kv_shared(x.q[idx], x.k_new[idx], sub(x.k_cache), sub(x.cap),
                                          sub(x.count_before), sub(x.is_ring), w, amp,
                                          q_gamma=gq, k_gamma=gk, eps=EPS, scale=scale)


def _check_decode(o, lse, e2e, what):
    _report(o, e2e[0], f"{what} (end to end)")
    _report(lse, e2e[1], f"{what} lse (end to end)")


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 2, 512), (16, 8, 256), (8, 1, 128), (6, 3, 256)])
def test_decode_kv_shared(Hq, Hkv, d):
    """Linear caches across split boundaries and rings around wrap-around; the new token's
    Z is normalised into its slot, the query normalised, then one decode step."""
    gu.require_gpu()
    x = _random_batch([0, 15, 1023, 1024, 2100], [(64, 10), (64, 200), (1024, 1023),
                                                  (1024, 3000)], Hq, Hkv, d, seed=1700 + d + Hq)
    x = replace(x, k_cache=[(t.float() * 3).to(torch.bfloat16) for t in x.k_cache])
    if d == 512:
        x = replace(x, rope=[PROPE if not r else LOCAL for r in x.is_ring])
    gq, gk = norm_gains(d, 1800 + d), norm_gains(d, 1900 + d)
    st = _shared_setup(x, d)
    o, lse, slots = _shared_step(st, x, Hq, Hkv, d, gq, gk, max_len=4096)
    e2e = _oracle_shared(x, d, gq, gk)
    _, _, rslots, rcounts = e2e
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), rslots)
    assert np.array_equal(st.counts(), rcounts)
    # the appended rows hold Zn of the new token; the decoy V caches are untouched
    rz = gu.orc().rms_norm(x.k_new, None, EPS)
    for i in range(x.q.shape[0]):
        for h in range(Hkv):
            gu.compare(st.kc[i][h, int(rslots[i])], rz[i, h], what=f"appended Zn {i}")
        assert torch.equal(st.vc[i].cpu(), x.v_cache[i])
    _check_decode(o, lse, e2e, f"kv-shared decode d={d} Hq={Hq} Hkv={Hkv}")


def test_decode_kv_shared_long_splits():
    """max_len 8192 with lengths at split boundaries, d = 512."""
    gu.require_gpu()
    Hq, Hkv, d = 16, 2, 512
    x = _random_batch([2047, 2048, 2049, 4100], [(1024, 3000)], Hq, Hkv, d, seed=2100)
    x = replace(x, k_cache=[(t.float() * 3).to(torch.bfloat16) for t in x.k_cache],
                rope=[PROPE if not r else LOCAL for r in x.is_ring])
    gq, gk = norm_gains(d, 2101), norm_gains(d, 2102)
    st = _shared_setup(x, d)
    o, lse, slots = _shared_step(st, x, Hq, Hkv, d, gq, gk, max_len=8192)
    e2e = _oracle_shared(x, d, gq, gk)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), e2e[2])
    assert np.array_equal(st.counts(), e2e[3])
    _check_decode(o, lse, e2e, "kv-shared decode, long caches")


def test_decode_kv_shared_equals_separate_caches():
    """The shared kernel over Zn equals the plain decode kernel over K = gamma_k Zn and
    V = Zn stored separately: the sharing changes which bytes are read, not the result.
    The gains are powers of two, so gamma_k Zn is exact in bf16 and the fp32 product the
    shared kernel forms is the same number as the stored key (built here with torch)."""
    gu.require_gpu()
    Hq, Hkv, d = 16, 2, 512
    x = _random_batch([700, 3000], [(1024, 2500)], Hq, Hkv, d, seed=2000)
    expo = torch.randint(-3, 2, (d,), generator=torch.Generator().manual_seed(2001))
    gk = torch.pow(2.0, expo.to(torch.float64)).numpy()
    st = _shared_setup(x, d)
    # separate caches made from the shared one
    gk_bf = torch.from_numpy(gk).to(torch.bfloat16).cuda()
    kc = [(zc * gk_bf).contiguous() for zc in st.kc]
    vc = [zc.clone() for zc in st.kc]
    a = gqa.make_kv_descs(kc, vc, [st.tables[r][0] for r in x.rope], x.cap,
                          [c + 1 for c in x.count_before], x.is_ring,
                          [st.tables[r][1] for r in x.rope])
    descs_sep = torch.from_numpy(a.view(np.uint8).copy()).cuda()
    a2 = gqa.make_kv_descs(st.kc, st.vc, [st.tables[r][0] for r in x.rope], x.cap,
                           [c + 1 for c in x.count_before], x.is_ring,
                           [st.tables[r][1] for r in x.rope])
    descs_sh = torch.from_numpy(a2.view(np.uint8).copy()).cuda()
    nseq, max_len = x.q.shape[0], 4096
    wsb = gqa.gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    o1, o2 = torch.empty_like(st.q), torch.empty_like(st.q)
    gqa.gqa_attn_decode(st.q, descs_sep, nseq, Hq, Hkv, d, 0.05, max_len, o1, None, ws, wsb)
    gqa.gqa_attn_decode_kv_shared(st.q, descs_sh, nseq, Hq, Hkv, d, 0.05, _dev_gain(gk),
                                  max_len, o2, None, ws, wsb)
    assert gqa.gqa_get_device_status() == 0
    assert torch.equal(o1, o2)


def test_gemma4_decode_global_kv_shared_full_size_sampled():
    """The benchmark's batch: 32 global caches of 8192..65536 tokens, d = 512, 2 KV heads,
    p-RoPE, one launch over every sequence; 6 sequences (the longest, the shortest and 4
    seeded others) compared with the oracle, all slots and counts bit-exact."""
    gu.require_gpu()
    w = get_workload("gemma4_decode_global_kv_shared")
    x = decode_inputs(w)
    gq, gk = norm_gains(w.d, w.seed + 1), norm_gains(w.d, w.seed + 2)
    st = _shared_setup(x, w.d)
    max_len = max(w.global_len_range[1], w.window)
    o, lse, slots = _shared_step(st, x, w.Hq, w.Hkv, w.d, gq, gk, max_len, w.scale)
    lens = np.array(x.count_before)
    rng = np.random.default_rng(11)
    idx = sorted({int(lens.argmax()), int(lens.argmin())} |
                 set(rng.choice(w.nseq, 4, replace=False).tolist()))
    e2e = _oracle_shared(x, w.d, gq, gk, idx, w.scale)
    rslots = e2e[2]
    want_slots = [gu.orc().append_slot(r, c, cap)
                  for r, c, cap in zip(x.is_ring, x.count_before, x.cap)]
    assert slots.cpu().tolist() == want_slots
    assert st.counts().tolist() == [c + 1 for c in x.count_before]
    assert rslots.tolist() == [want_slots[i] for i in idx]
    _check_decode(o[idx], lse[idx], e2e, "gemma4 kv-shared decode (sampled sequences)")
