"""The debug build: the library compiled with GQA_DEBUG_BOUNDS, in which every global access
whose index comes from device-side data (cache slots and counts from the descriptors,
RoPE table rows, split-KV workspace records) is checked before it is made; a failed check
records GQA_ERR_DEVICE_BOUNDS and skips the access instead of touching memory out of
range.  It stands in for a memory checker.

The test builds that library into its own file (libgqa_attn_debug.so), loads it in place
of the normal one for this module, and runs the decode, shared K/V, chunked prefill, Q/K
normalisation and prefill parity cases on their odd and tiny shapes through it: every
output still matches the fp64 oracle and the device status stays 0, so no check fires.
"""
import pytest

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
import test_gpu_chunked as t_chunk
import test_gpu_decode as t_dec
import test_gpu_kv_shared as t_kvs
import test_gpu_prefill as t_pf
import test_gpu_qknorm as t_qk
from global_causal_gqa_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    gu.require_gpu()
    path = build.build(debug=True)
    saved_path, saved_lib = gqa.LIB_PATH, gqa._lib
    gqa.LIB_PATH, gqa._lib = path, None
    try:
        assert gqa.lib()._name == path
        assert gqa.gqa_get_device_status() == 0
        yield path
    finally:
        gqa.LIB_PATH, gqa._lib = saved_path, saved_lib


def _clean():
    st = gqa.gqa_get_device_status()
    assert st == 0, gqa.STATUS_NAMES.get(st, st)


def test_decode_in_debug_build(debug_lib):
    t_dec.test_mixed_small_batch(6, 2)
    t_dec.test_mixed_small_batch(8, 1)
    t_dec.test_wide_head_decode(6, 3, 256)
    t_dec.test_wide_head_decode(16, 2, 512)
    t_dec.test_odd_partial_counts(3, 7, 1, 128, 448)
    t_dec.test_odd_partial_counts(1, 3, 1, 512, 320)
    t_dec.test_long_split_boundaries(16, 2)
    t_dec.test_two_steps_in_a_row()
    t_dec.test_cache_rows_written_exactly()
    _clean()


def test_shared_kv_in_debug_build(debug_lib):
    t_kvs.test_decode_kv_shared(6, 3, 256)
    t_kvs.test_decode_kv_shared(8, 1, 128)
    t_kvs.test_prefill_kv_shared(128, 6, 3, 200, 64, t_dec.LOCAL)
    _clean()


def test_chunked_and_norm_in_debug_build(debug_lib):
    t_chunk.test_chunks_3_6_3_equal_one_pass(256, t_chunk.LOCAL, 256)
    t_chunk.test_chunks_3_6_3_equal_one_pass(0, t_chunk.YARN, None)
    t_chunk.test_ring_chunk_longer_than_ring_keeps_last_tokens()
    t_qk.test_decode_norm_append_then_attend(0)
    t_qk.test_decode_norm_append_then_attend(1)
    t_qk.test_prefill_norm_then_rope(256, t_qk.RopeSpec(base=1e4), 5)
    _clean()


@pytest.mark.parametrize("layer", t_pf.EDGE_CASES[:8] + t_pf.WIDE_CASES[:4] + t_pf.WIDE_CASES[10:],
                         ids=lambda l: l.label)
def test_prefill_in_debug_build(debug_lib, layer):
    t_pf._full_case(layer)
    _clean()
