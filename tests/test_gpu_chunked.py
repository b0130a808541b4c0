"""Chunked prefill over a KV cache: gqa_prefill_gather + gqa_attn_prefill +
gqa_kv_append_chunk, chunk after chunk, against the fp64 oracle's one-pass prefill.

The pages check that a sequence processed in chunks (3/6/3 tokens) gives the outputs of
one pass; here a 1536-token sequence goes in chunks of 384/768/384.  A local layer keeps
a ring of W = 256 tokens and re-numbers positions from 0 (RoPE depends only on position
differences, so the outputs equal the one-pass ones at absolute positions); a global
layer keeps a linear cache.  Cache slots after the appends are checked bit-exactly
against the oracle's cache index model.
"""
import math

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from workloads import RopeSpec

pytestmark = pytest.mark.gpu

LOCAL = RopeSpec(base=1e4)
YARN = RopeSpec(base=1e6, yarn_factor=8.0, amp=math.sqrt(1.2))


def _chunked(N, chunks, Hq, Hkv, d, window, rope, ring_cap, seed):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    q, k, v = bf(1, Hq, N, d), bf(1, Hkv, N, d), bf(1, Hkv, N, d)
    scale = 1 / math.sqrt(d)
    cap = ring_cap if ring_cap else N
    table_len = N + (ring_cap or 0)
    table = gu.rope_table(d, rope, table_len)
    kc = torch.zeros(Hkv, cap, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    a = gqa.make_kv_descs([kc], [vc], [table], [cap], [0], [1 if ring_cap else 0], [table_len])
    desc = torch.from_numpy(a.view(np.uint8).copy()).cuda()
    outs, count = [], 0
    pos = 0
    for T in chunks:
        R = min(count, cap) if ring_cap else count
        S = R + T
        kn = k[0, :, pos:pos + T].contiguous().cuda()
        vn = v[0, :, pos:pos + T].contiguous().cuda()
        k_lin = torch.empty(Hkv, S, d, dtype=torch.bfloat16, device="cuda")
        v_lin = torch.empty_like(k_lin)
        gqa.gqa_prefill_gather(desc, kn, vn, T, Hkv, d, k_lin, v_lin, S, table, table_len)
        qc = q[:, :, pos:pos + T].contiguous().cuda()
        o = torch.empty_like(qc)
        lse = torch.empty(1, Hq, T, dtype=torch.float32, device="cuda")
        gqa.gqa_attn_prefill(qc, k_lin, v_lin, o, lse, 1, T, S, Hq, Hkv, d, window, scale,
                             table, table_len, 1, None, 0)
        gqa.gqa_kv_append_chunk(desc, 1, kn, vn, T, Hkv, d)
        st = gqa.gqa_get_device_status()
        assert st == 0, gqa.STATUS_NAMES.get(st, st)
        outs.append(o.cpu())
        count += T
        pos += T
    return q, k, v, torch.cat(outs, dim=2), kc, vc, desc, count, cap


@pytest.mark.parametrize("window,rope,ring_cap", [(256, LOCAL, 256), (0, YARN, None)])
def test_chunks_3_6_3_equal_one_pass(window, rope, ring_cap):
    gu.require_gpu()
    N, chunks, Hq, Hkv, d = 1536, (384, 768, 384), 8, 2, 128
    q, k, v, o, kc, vc, desc, count, cap = _chunked(N, chunks, Hq, Hkv, d, window, rope,
                                                    ring_cap, seed=1100 + window)
    orc = gu.orc()
    ro, _ = orc.attention(q, k, v, window=window, scale=1 / math.sqrt(d),
                          w=gu.oracle_freq(d, rope), amp=rope.amp)
    gu.compare(o, ro, what=f"chunked W={window}")
    # the cache after the appends: logical token t of the retained ones sits where the
    # oracle's index model puts it, bit for bit
    is_ring = 1 if ring_cap else 0
    R = orc.retained(is_ring, count, cap)
    kh, vh = kc.cpu(), vc.cpu()
    for t in range(R):
        slot = orc.logical_slot(is_ring, count, cap, t)
        tok = count - R + t
        assert torch.equal(kh[:, slot], k[0, :, tok]) and torch.equal(vh[:, slot], v[0, :, tok])
    assert desc.cpu().numpy().view(gqa.KV_DESC_DTYPE)["count"][0] == count


def test_ring_chunk_longer_than_ring_keeps_last_tokens():
    gu.require_gpu()
    Hkv, d, cap, T = 2, 128, 64, 150
    g = torch.Generator().manual_seed(1200)
    kn = torch.randn(1, Hkv, T, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(1, Hkv, T, d, generator=g).to(torch.bfloat16)
    kc = torch.zeros(Hkv, cap, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    tab = gu.rope_table(d, LOCAL, 8)
    a = gqa.make_kv_descs([kc], [vc], [tab], [cap], [37], [1], [8])
    desc = torch.from_numpy(a.view(np.uint8).copy()).cuda()
    gqa.gqa_kv_append_chunk(desc, 1, kn.cuda(), vn.cuda(), T, Hkv, d)
    assert gqa.gqa_get_device_status() == 0
    orc = gu.orc()
    after = 37 + T
    for t in range(cap):
        slot = orc.logical_slot(1, after, cap, t)
        tok = T - cap + t
        assert torch.equal(kc[:, slot].cpu(), kn[0, :, tok])
        assert torch.equal(vc[:, slot].cpu(), vn[0, :, tok])


def test_gather_rejects_wrong_length_and_full_linear_cache():
    gu.require_gpu()
    Hkv, d = 1, 128
    kc = torch.zeros(Hkv, 32, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    tab = gu.rope_table(d, LOCAL, 64)
    a = gqa.make_kv_descs([kc], [vc], [tab], [32], [20], [0], [64])
    desc = torch.from_numpy(a.view(np.uint8).copy()).cuda()
    kn = torch.zeros(Hkv, 16, d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(Hkv, 40, d, dtype=torch.bfloat16, device="cuda")
    # the descriptor holds 20 tokens: S must be 36, not 40
    gqa.gqa_prefill_gather(desc, kn, kn, 16, Hkv, d, out, out, 40, tab, 64)
    assert gqa.gqa_get_device_status() == -4
    assert torch.count_nonzero(out).item() == 0
    # 20 + 16 > 32: the linear cache refuses the chunk and keeps its count
    gqa.gqa_kv_append_chunk(desc, 1, kn.unsqueeze(0).contiguous(), kn.unsqueeze(0).contiguous(),
                            16, Hkv, d)
    assert gqa.gqa_get_device_status() == -4
    assert desc.cpu().numpy().view(gqa.KV_DESC_DTYPE)["count"][0] == 20
