"""The 64-layer PLaMo-3-shaped decode step (7 ring layers of W = 2048 then 1 linear global
layer of N = 4096 tokens, per period; "PLaMo 3アーキテクチャ徹底解析" §2.3, §4.4) against the
oracle, built exactly as the benchmark builds and times it (bench.decode_model_stack):
one descriptor buffer for every layer, append + decode per layer, run eagerly and as a
replayed CUDA graph whose first node restores every layer's counts.

Sampled: a ring layer at the start, the global layer of the first period, a ring layer in
the middle and the last (global) layer, three sequences of each, compared with the fp64
oracle's decode step over the caches as they were before the step (max abs 2e-2, mean
abs 2e-3; slots and counts bit-exact).  Every layer's counts are checked after each run,
and the graph replays -- which restore the counts and append into the same slots again --
must reproduce the eager step bit for bit.
"""
import numpy as np
import pytest
import torch

import bench
import gpu_utils as gu
from workloads import get_workload
from workloads.gen import DecodeInputs

pytestmark = pytest.mark.gpu

LAYERS = (0, 7, 30, 63)
SEQS = (0, 13, 31)


def test_plamo3_decode_64layer_step_sampled():
    gu.require_gpu()
    import global_causal_gqa_gb300 as gqa
    w = get_workload("plamo3_decode_64layer")
    stack = bench.decode_model_stack(w)
    seqs = list(SEQS)
    # the sampled layers' state before the step, on the host
    before = {}
    for l in LAYERS:
        L = stack.layers[l]
        before[l] = DecodeInputs(
            L.q[seqs].cpu(), L.k_new[seqs].cpu(), L.v_new[seqs].cpu(),
            [L.k_cache[i].cpu() for i in seqs], [L.v_cache[i].cpu() for i in seqs],
            [L.k_cache.shape[2]] * len(seqs), [L.count_before[i] for i in seqs],
            [int(L.is_ring)] * len(seqs),
            [w.rope_local if L.is_ring else w.rope_global] * len(seqs))
    want = [np.array(L.count_before, dtype=np.int64) + 1 for L in stack.layers]

    stack.step()
    torch.cuda.synchronize()
    assert gqa.gqa_get_device_status() == 0
    eager = {l: stack.layers[l].o.clone() for l in LAYERS}
    for l in range(w.layers):
        assert np.array_equal(stack.counts(l), want[l]), l

    graph = stack.capture()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert gqa.gqa_get_device_status() == 0
        for l in range(w.layers):
            assert np.array_equal(stack.counts(l), want[l]), l
        for l in LAYERS:
            assert torch.equal(stack.layers[l].o, eager[l]), l

    orc = gu.orc()
    for l in LAYERS:
        x = before[l]
        fw = [gu.oracle_freq(w.d, r) for r in x.rope]
        ro, rl, rslots, rcounts = orc.decode_step(x.q, x.k_new, x.v_new, x.k_cache, x.v_cache,
                                                  x.cap, x.count_before, x.is_ring, fw,
                                                  [r.amp for r in x.rope], w.scale)
        assert np.array_equal(rcounts, want[l][seqs])
        slot = [orc.append_slot(r, c, cap) for r, c, cap in zip(x.is_ring, x.count_before,
                                                                   x.cap)]
        assert rslots.tolist() == slot
        L = stack.layers[l]
        for j, i in enumerate(seqs):   # the appended rows landed in those slots
            assert torch.equal(L.k_cache[i][:, slot[j]].cpu(), x.k_new[j])
            assert torch.equal(L.v_cache[i][:, slot[j]].cpu(), x.v_new[j])
        gu.compare(eager[l][seqs], ro, what=f"64-layer step, layer {l}")
