"""Failure detection on the GPU without a fault.

Every wait in the kernels is bounded; when one expires the kernel records
GQA_ERR_DEVICE_TIMEOUT with a diagnostic code and returns.  gqa_watchdog_selftest runs
that same wait-and-report code on an mbarrier nothing arrives on, so the wait must
expire.  The tests check the status and code the host reads back, that reading clears
them, that the wait lasted about as long as asked, and that the context is still usable
afterwards (a prefill right after it matches the oracle).
"""
import time

import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from workloads import WORKLOADS

pytestmark = pytest.mark.gpu

TIMEOUT = -6
WATCHDOG_CODE = 4 << 24


def _clear():
    gqa.gqa_get_device_diag()
    gqa.gqa_get_device_status()


def test_expired_wait_is_reported_and_cleared():
    gu.require_gpu()
    _clear()
    assert gqa.gqa_get_device_status() == 0
    t0 = time.perf_counter()
    gqa.gqa_watchdog_selftest(200_000_000)        # 0.2 s
    st = gqa.gqa_get_device_status()
    dt = time.perf_counter() - t0
    assert st == TIMEOUT
    assert 0.19 <= dt < 5.0, dt
    diag = gqa.gqa_get_device_diag()
    assert diag[0] == WATCHDOG_CODE and diag[1] == WATCHDOG_CODE, diag
    assert diag[2:] == [0, 0, 0]
    # both were cleared by the reads
    assert gqa.gqa_get_device_status() == 0
    assert gqa.gqa_get_device_diag() == [0, 0, 0, 0, 0]


def test_context_usable_after_expired_waits():
    gu.require_gpu()
    _clear()
    s = torch.cuda.Stream()
    for _ in range(3):
        gqa.gqa_watchdog_selftest(20_000_000, stream=s)   # 20 ms each, queued back to back
    assert gqa.gqa_get_device_status(stream=s) == TIMEOUT
    _clear()
    layer = WORKLOADS["tiny_w64"].layers[0]
    from workloads import prefill_inputs
    x = prefill_inputs(layer)
    q, k, v = gu.to_cuda(x.q, x.k, x.v)
    table = gu.rope_table(layer.d, layer.rope, layer.S)
    o, _ = gu.run_prefill(q, k, v, layer.window, layer.scale, table, layer.S)
    assert gqa.gqa_get_device_status() == 0
    ro, _ = gu.orc().attention(x.q, x.k, x.v, window=layer.window, scale=layer.scale,
                               w=gu.oracle_freq(layer.d, layer.rope), amp=layer.rope.amp)
    gu.compare(o, ro, what="prefill after watchdog")
