"""Q/K normalisation in front of attention (gqa_qk_norm_rope, gqa_qk_norm_append)
against the fp64 oracle.

RMSNorm with an effective gain (offset 1 plus a stored weight), eps 1e-6, one gain of d
values shared by every head; the prefill form also rotates the normalised K (norm first,
then RoPE, the order the pages fix), the decode form appends the normalised K and the
projected V to the cache.  Bar: max abs 2e-2 / mean abs 2e-3 on the bf16 outputs; slots
and counts bit-exact.
"""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from test_gpu_decode import LOCAL, YARN, DecodeSetup, _random_batch, oracle_step
from workloads import RopeSpec

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _bf(shape, g):
    return torch.randn(*shape, generator=g).to(torch.bfloat16)


def _gain(d, seed):
    g = torch.Generator().manual_seed(seed)
    return (1.0 + 0.2 * torch.randn(d, generator=g, dtype=torch.float64)).numpy()


def _to_bf16_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a).to(torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("d,rope,pos0", [(64, LOCAL, 0), (128, LOCAL, 0), (128, YARN, 37),
                                         (256, RopeSpec(base=1e4), 5),
                                         (512, RopeSpec(base=1e6, rotate_fraction=0.25), 0)])
def test_prefill_norm_then_rope(d, rope, pos0):
    gu.require_gpu()
    B, Hq, Hkv, T = 2, 6, 2, 77
    g = torch.Generator().manual_seed(900 + d + pos0)
    q, k = _bf((B, Hq, T, d), g), _bf((B, Hkv, T, d), g)
    k = (k.to(torch.float32) * 3).to(torch.bfloat16)          # any scale: RMSNorm removes it
    gq, gk = _gain(d, 1), _gain(d, 2)
    table = gu.rope_table(d, rope, pos0 + T)
    qd, kd = q.cuda(), k.cuda()
    q_out, k_out, k_rot = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(kd)
    gqd = torch.from_numpy(gq).to(torch.float32).cuda()
    gkd = torch.from_numpy(gk).to(torch.float32).cuda()
    gqa.gqa_qk_norm_rope(qd, kd, q_out, k_out, k_rot, B, Hq, Hkv, T, d, pos0, gqd, gkd, EPS,
                         table, pos0 + T)
    assert gqa.gqa_get_device_status() == 0
    orc = gu.orc()
    # the oracle takes the same fp32 gains the device reads
    gq32, gk32 = gq.astype(np.float32).astype(np.float64), gk.astype(np.float32).astype(np.float64)
    rq, rk = orc.rms_norm(q, gq32, EPS), orc.rms_norm(k, gk32, EPS)
    gu.compare(q_out, rq, what="q_out")
    gu.compare(k_out, rk, what="k_out")
    w = gu.oracle_freq(d, rope)
    rrot = np.empty_like(rk)
    wrong = np.empty_like(rk)
    kk = k.to(torch.float64).numpy()
    for b in range(B):
        for h in range(Hkv):
            for t in range(T):
                rrot[b, h, t] = orc.rope_rotate(rk[b, h, t], pos0 + t, w, rope.amp)
                # the other order: rotate, then normalise (the pages: not the same vector)
                x = orc.rope_rotate(kk[b, h, t], pos0 + t, w, rope.amp)
                wrong[b, h, t] = gk32 * x / math.sqrt(np.mean(x * x) + EPS)
    gu.compare(k_rot, rrot, what="k_rot")
    if rope.rotate_fraction == 1.0 and rope.base < 1e6:
        err = np.abs(k_rot.float().cpu().numpy() - wrong).max()
        assert err > 0.1, "norm-then-rotate should differ from rotate-then-norm"


def test_prefill_in_place_and_optional_outputs():
    gu.require_gpu()
    B, Hq, Hkv, T, d = 1, 4, 1, 40, 128
    g = torch.Generator().manual_seed(950)
    q, k = _bf((B, Hq, T, d), g), _bf((B, Hkv, T, d), g)
    gq = torch.ones(d, dtype=torch.float32, device="cuda")
    gk = torch.full((d,), 0.5, dtype=torch.float32, device="cuda")
    qd, kd = q.cuda(), k.cuda()
    gqa.gqa_qk_norm_rope(qd, kd, qd, kd, None, B, Hq, Hkv, T, d, 0, gq, gk, EPS, None, 0)
    assert gqa.gqa_get_device_status() == 0
    orc = gu.orc()
    gu.compare(qd, orc.rms_norm(q, np.ones(d), EPS), what="q in place")
    gu.compare(kd, orc.rms_norm(k, np.full(d, 0.5), EPS), what="k in place")


@pytest.mark.parametrize("v_norm", [0, 1])
def test_decode_norm_append_then_attend(v_norm):
    """Normalise and append one token per sequence, then decode: equal to the oracle's
    decode step on the oracle-normalised inputs (rounded to bf16, the cache's format)."""
    gu.require_gpu()
    Hq, Hkv, d = 16, 2, 128
    x = _random_batch([30, 700, 0], [(64, 63), (64, 200), (128, 5)], Hq, Hkv, d, seed=960)
    gq, gk = _gain(d, 3), _gain(d, 4)
    gq32, gk32 = gq.astype(np.float32).astype(np.float64), gk.astype(np.float32).astype(np.float64)
    st = DecodeSetup(x, d)
    nseq = x.q.shape[0]
    q_out = torch.empty_like(st.q)
    slots = torch.full((nseq,), -7, dtype=torch.int32, device="cuda")
    gqa.gqa_qk_norm_append(st.descs, nseq, st.q, st.k_new, st.v_new, Hq, Hkv, d,
                           torch.from_numpy(gq).float().cuda(), torch.from_numpy(gk).float().cuda(),
                           EPS, v_norm, q_out, slots)
    o = torch.empty_like(st.q)
    max_len = 1024
    wsb = gqa.gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    scale = 1 / math.sqrt(d)
    gqa.gqa_attn_decode(q_out, st.descs, nseq, Hq, Hkv, d, scale, max_len, o, None, ws, wsb)
    assert gqa.gqa_get_device_status() == 0
    orc = gu.orc()
    # slots and counts: the cache index model, bit-exact
    want_slots = [orc.append_slot(r, c, cap) for r, c, cap in zip(x.is_ring, x.count_before, x.cap)]
    assert slots.cpu().tolist() == want_slots
    assert st.counts().tolist() == [c + 1 for c in x.count_before]
    rq = orc.rms_norm(x.q, gq32, EPS)
    rk = orc.rms_norm(x.k_new, gk32, EPS)
    rv = orc.rms_norm(x.v_new, None, EPS) if v_norm else x.v_new.to(torch.float64).numpy()
    gu.compare(q_out, rq, what="q_out")
    # the appended rows in the caches
    for i in range(nseq):
        for h in range(Hkv):
            gu.compare(st.kc[i][h, want_slots[i]], rk[i, h], what=f"k row {i}")
            gu.compare(st.vc[i][h, want_slots[i]], rv[i, h], what=f"v row {i}")
    # attention over the normalised token: the oracle's decode on bf16-rounded inputs
    xn = replace(x, q=_to_bf16_bits(rq), k_new=_to_bf16_bits(rk), v_new=_to_bf16_bits(rv))
    ro, _, _, _ = oracle_step(xn, d, scale)
    gu.compare(o, ro, what="decode after norm+append")


def test_norm_append_full_linear_cache_is_reported():
    gu.require_gpu()
    Hq, Hkv, d = 8, 1, 128
    x = _random_batch([16], [], Hq, Hkv, d, seed=970)
    x.cap[0] = 16           # already full
    st = DecodeSetup(x, d)
    one = torch.ones(d, dtype=torch.float32, device="cuda")
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    gqa.gqa_qk_norm_append(st.descs, 1, st.q, st.k_new, st.v_new, Hq, Hkv, d, one, one, EPS, 0,
                           torch.empty_like(st.q), slots)
    assert gqa.gqa_get_device_status() == -4          # GQA_ERR_CAPACITY
    assert slots.cpu().tolist() == [-1] and st.counts().tolist() == [16]
