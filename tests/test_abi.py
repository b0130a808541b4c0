"""The C-ABI library without a GPU: it loads, exports every function the header declares,
its host-only functions agree with the oracle, and bad arguments are rejected on the
host before anything is launched."""
import math
import os
import re

import numpy as np
import pytest

import global_causal_gqa_gb300 as gqa
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "gqa_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = gqa.lib()
    names = _declared()
    assert len(names) >= 13, names
    for n in names:
        assert hasattr(L, n), n


def test_inv_freq_matches_oracle():
    orc = oracle.default()
    for args in [(128, 1e4), (128, 1e6, 8.0), (128, 1e6, 256.0), (512, 1e6, 1.0, 4096, 32, 1, 0.25),
                 (256, 1e4), (64, 5e5, 4.0, 8192, 16, 2)]:
        a = gqa.gqa_rope_inv_freq(*args)
        b = orc.inv_freq(*args)
        assert np.max(np.abs(a - b)) <= 1e-15 * np.max(np.abs(b)), args


def test_yarn_amplitude_and_sizes():
    assert abs(gqa.gqa_yarn_amplitude(256.0) - (1 + 0.1 * math.log(256))) < 1e-15
    assert gqa.gqa_rope_table_bytes(128, 1000) == 1000 * 64 * 2 * 4
    assert gqa.gqa_prefill_workspace_bytes(2, 8, 8192, 128) == 2 * 8 * 8192 * 128 * 2
    # decode: a whole number of splits per (sequence, query head), each a partial of d + 2
    # floats, at least one split and no more than one per 16 keys
    for args in [(32, 64, 8, 128, 65536), (32, 16, 8, 256, 1024), (2, 8, 1, 512, 4097),
                 (1, 1, 1, 128, 1)]:
        nseq, Hq, Hkv, d, max_len = args
        total = gqa.gqa_decode_workspace_bytes(*args)
        ns = (total // 4) // (nseq * Hq * (d + 2))
        assert 1 <= ns <= -(-max_len // 16), args
        assert total == 4 * (-(-2 * nseq * Hq * ns // 4) * 4 + nseq * Hq * ns * d), args
    assert gqa.gqa_decode_workspace_bytes(2, 8, 0, 128, 64) == 0
    assert gqa.gqa_rope_table_bytes(0, 10) == 0


def test_decode_workspace_layout_keeps_partials_aligned():
    """The decode workspace holds nseq*Hq*nsplit (m, l) float pairs, then the O partials,
    which the kernel writes with 16-byte stores.  For odd nseq*Hq*nsplit the pairs take an
    odd number of 8-byte slots, so the O rows would start 8 bytes off a 16-byte boundary
    unless the pairs are padded: the bytes before the O rows (the total minus the O rows'
    nseq*Hq*nsplit*d floats) must be a multiple of 16 and hold the pairs with at most 8
    bytes of padding."""
    for nseq in (1, 2, 3, 5, 31):
        for Hq in (1, 2, 3, 5, 7, 64):
            for d in (128, 256, 512):
                for max_len in (1, 256, 257, 768, 1280, 4096, 4097, 6145, 65536):
                    Hkv = 1
                    total = gqa.gqa_decode_workspace_bytes(nseq, Hq, Hkv, d, max_len)
                    ns = (total // 4) // (nseq * Hq * (d + 2))   # splits per sequence
                    head = total - nseq * Hq * ns * d * 4
                    pairs = 2 * nseq * Hq * ns * 4
                    assert head % 16 == 0, (nseq, Hq, d, max_len)
                    assert pairs <= head <= pairs + 8, (nseq, Hq, d, max_len)


def test_non_positive_scale_rejected_on_host():
    """The kernels take each row's maximum score before scaling, which is only the
    maximum of the scaled scores for scale > 0: every attention call rejects others."""
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    fake = 0x10000
    wsb = gqa.gqa_decode_workspace_bytes(1, 2, 1, 128, 64)
    for bad in (0.0, -0.125, float("-inf"), float("nan")):
        assert S[L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 2, 1, 128, 0, bad,
                                    fake, 8, 1, None, 0, None)] == "GQA_ERR_INVALID_ARG"
        assert S[L.gqa_attn_decode(fake, fake, 1, 2, 1, 128, bad, 64, fake, None, fake, wsb,
                                   None)] == "GQA_ERR_INVALID_ARG"
        assert S[L.gqa_attn_decode_kv_shared(fake, fake, 1, 2, 1, 128, bad, fake, 64, fake,
                                             None, fake, wsb, None)] == "GQA_ERR_INVALID_ARG"
        assert S[L.gqa_attn_decode_static(fake, fake, 1, 2, 1, 128, bad, 64, fake, None,
                                          None)] == "GQA_ERR_INVALID_ARG"


def test_bad_arguments_rejected_on_host():
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    f = lambda st: S.get(st, st)  # noqa: E731
    with pytest.raises(gqa.GQAError):
        gqa.gqa_rope_inv_freq(127, 1e4)
    # null pointers
    assert f(L.gqa_attn_prefill(None, None, None, None, None, 1, 8, 8, 2, 1, 128, 0, 0.1,
                                None, 8, 0, None, 0, None)) == "GQA_ERR_INVALID_ARG"
    fake = 0x10000
    # T > S, Hq not a multiple of Hkv
    assert f(L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 9, 8, 2, 1, 128, 0, 0.1, fake,
                                8, 0, fake, 1 << 20, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 3, 2, 128, 0, 0.1, fake,
                                8, 0, fake, 1 << 20, None)) == "GQA_ERR_INVALID_ARG"
    # unsupported head dim, misaligned pointer, short table, small workspace
    assert f(L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 2, 1, 96, 0, 0.1, fake,
                                8, 0, fake, 1 << 20, None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_attn_prefill(fake + 8, fake, fake, fake, None, 1, 8, 8, 2, 1, 128, 0, 0.1,
                                fake, 8, 0, fake, 1 << 20, None)) == "GQA_ERR_ALIGNMENT"
    assert f(L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 2, 1, 128, 0, 0.1, fake,
                                7, 0, fake, 1 << 20, None)) == "GQA_ERR_RANGE"
    assert f(L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 2, 1, 128, 0, 0.1, fake,
                                8, 0, fake, 10, None)) == "GQA_ERR_WORKSPACE"
    # decode: group larger than supported, small workspace
    assert f(L.gqa_attn_decode(fake, fake, 1, 32, 2, 128, 0.1, 64, fake, None, fake, 1 << 20,
                               None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_attn_decode(fake, fake, 1, 8, 1, 128, 0.1, 64, fake, None, fake, 8,
                               None)) == "GQA_ERR_WORKSPACE"
    assert f(L.gqa_kv_append(None, 1, fake, fake, 1, 128, None, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_rope_apply(fake, fake, 1, 1, 4, 128, 10, fake, 12, None)) == "GQA_ERR_RANGE"
    assert gqa.gqa_status_string(-6) == "device-side wait timed out"


def test_k_rotation_modes_checked_on_host():
    """k_is_rotated: 0 (rotate once into the workspace), 1 (already rotated), 2 (rotated in
    the tile load, d = 128 only); anything else is rejected before any launch."""
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    fake = 0x10000
    for bad in (-1, 3, 7):
        assert S[L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 2, 1, 128, 0, 0.1,
                                    fake, 8, bad, None, 0, None)] == "GQA_ERR_INVALID_ARG"
    for d in (256, 512):
        assert S[L.gqa_attn_prefill(fake, fake, fake, fake, None, 1, 8, 8, 2, 1, d, 0, 0.1,
                                    fake, 8, 2, None, 0, None)] == "GQA_ERR_UNSUPPORTED"


def test_watchdog_selftest_limits_rejected_on_host():
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    for bad in (0, 999, -5, 2_000_000_001):
        assert S[L.gqa_watchdog_selftest(bad, None)] == "GQA_ERR_INVALID_ARG", bad


def test_qk_norm_arguments_rejected_on_host():
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    f = lambda st: S.get(st, st)  # noqa: E731
    fake = 0x10000
    # null gain, unsupported d, misaligned output, position past the table, bad v_norm
    assert f(L.gqa_qk_norm_rope(fake, fake, fake, None, None, 1, 2, 1, 8, 128, 0, None, fake,
                                1e-6, None, 0, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_qk_norm_rope(fake, fake, fake, None, None, 1, 2, 1, 8, 96, 0, fake, fake,
                                1e-6, None, 0, None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_qk_norm_rope(fake, fake, fake + 4, None, None, 1, 2, 1, 8, 128, 0, fake,
                                fake, 1e-6, None, 0, None)) == "GQA_ERR_ALIGNMENT"
    assert f(L.gqa_qk_norm_rope(fake, fake, fake, None, fake, 1, 2, 1, 8, 128, 3, fake, fake,
                                1e-6, fake, 10, None)) == "GQA_ERR_RANGE"
    assert f(L.gqa_qk_norm_append(fake, 1, fake, fake, fake, 2, 1, 128, fake, fake, 1e-6, 2,
                                  fake, None, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_qk_norm_append(fake, 1, fake, fake, fake, 2, 1, 128, fake, fake, -1.0, 0,
                                  fake, None, None)) == "GQA_ERR_INVALID_ARG"


def test_kv_shared_arguments_rejected_on_host():
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    f = lambda st: S.get(st, st)  # noqa: E731
    fake = 0x10000
    # prefill form: neither output, k_rot without its gain, q without q_out, misaligned
    # v_out, unsupported d, a position past the table
    assert f(L.gqa_qk_norm_rope_kv_shared(None, fake, None, None, None, 1, 0, 1, 8, 128, 0,
                                          None, fake, 1e-6, fake, 8, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_qk_norm_rope_kv_shared(None, fake, None, None, fake, 1, 0, 1, 8, 128, 0,
                                          None, None, 1e-6, fake, 8, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_qk_norm_rope_kv_shared(fake, fake, None, fake, None, 1, 2, 1, 8, 128, 0,
                                          fake, None, 1e-6, None, 0, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_qk_norm_rope_kv_shared(None, fake, None, fake + 8, None, 1, 0, 1, 8, 128, 0,
                                          None, None, 1e-6, None, 0, None)) == "GQA_ERR_ALIGNMENT"
    assert f(L.gqa_qk_norm_rope_kv_shared(None, fake, None, fake, None, 1, 0, 1, 8, 100, 0,
                                          None, None, 1e-6, None, 0, None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_qk_norm_rope_kv_shared(None, fake, None, None, fake, 1, 0, 1, 8, 128, 5,
                                          None, fake, 1e-6, fake, 12, None)) == "GQA_ERR_RANGE"
    # decode form: missing query gain, negative eps
    assert f(L.gqa_kv_shared_append(fake, 1, fake, fake, 2, 1, 128, None, 1e-6, fake, None,
                                    None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_kv_shared_append(fake, 1, fake, fake, 2, 1, 128, fake, -1.0, fake, None,
                                    None)) == "GQA_ERR_INVALID_ARG"
    # decode: no key gain, head dim 64, group of 16, too little workspace, misaligned gain
    wsb = gqa.gqa_decode_workspace_bytes(1, 2, 1, 128, 64)
    assert f(L.gqa_attn_decode_kv_shared(fake, fake, 1, 2, 1, 128, 1.0, None, 64, fake, None,
                                         fake, wsb, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_attn_decode_kv_shared(fake, fake, 1, 2, 1, 64, 1.0, fake, 64, fake, None,
                                         fake, wsb, None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_attn_decode_kv_shared(fake, fake, 1, 16, 1, 128, 1.0, fake, 64, fake, None,
                                         fake, wsb, None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_attn_decode_kv_shared(fake, fake, 1, 2, 1, 128, 1.0, fake, 64, fake, None,
                                         fake, wsb - 4, None)) == "GQA_ERR_WORKSPACE"
    assert f(L.gqa_attn_decode_kv_shared(fake, fake, 1, 2, 1, 128, 1.0, fake + 4, 64, fake, None,
                                         fake, wsb, None)) == "GQA_ERR_ALIGNMENT"


def test_chunked_prefill_arguments_rejected_on_host():
    L = gqa.lib()
    S = gqa.STATUS_NAMES
    f = lambda st: S.get(st, st)  # noqa: E731
    fake = 0x10000
    # S < T, unsupported d, misaligned output, S past the table
    assert f(L.gqa_prefill_gather(fake, fake, fake, 8, 1, 128, fake, fake, 4, fake, 64,
                                  None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_prefill_gather(fake, fake, fake, 8, 1, 96, fake, fake, 16, fake, 64,
                                  None)) == "GQA_ERR_UNSUPPORTED"
    assert f(L.gqa_prefill_gather(fake, fake, fake, 8, 1, 128, fake + 8, fake, 16, fake, 64,
                                  None)) == "GQA_ERR_ALIGNMENT"
    assert f(L.gqa_prefill_gather(fake, fake, fake, 8, 1, 128, fake, fake, 65, fake, 64,
                                  None)) == "GQA_ERR_RANGE"
    assert f(L.gqa_kv_append_chunk(fake, 1, fake, fake, 0, 1, 128, None)) == "GQA_ERR_INVALID_ARG"
    assert f(L.gqa_kv_append_chunk(fake + 4, 1, fake, fake, 4, 1, 128, None)) == "GQA_ERR_ALIGNMENT"
