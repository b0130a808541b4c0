"""RoPE table and rotation kernels against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import global_causal_gqa_gb300 as gqa
import gpu_utils as gu
from workloads import RopeSpec, randn_bf16

pytestmark = pytest.mark.gpu

SPECS = [RopeSpec(base=1e4), RopeSpec(base=1e6, yarn_factor=8.0, amp=math.sqrt(1.2)),
         RopeSpec(base=1e6, yarn_factor=256.0, amp=1.0 + 0.1 * math.log(256.0)),
         RopeSpec(base=1e6, rotate_fraction=0.25)]


@pytest.mark.parametrize("d,spec", [(128, s) for s in SPECS[:3]] + [(512, SPECS[3]), (256, SPECS[0])])
def test_table_matches_fp64(d, spec):
    """Each entry is amp*cos / amp*sin of p*omega_j rounded once to float32."""
    gu.require_gpu()
    P = 70000
    tab = gu.rope_table(d, spec, P).cpu().numpy().reshape(P, d // 2, 2).astype(np.float64)
    w = gu.oracle_freq(d, spec)
    for p in (0, 1, 2, 2047, 4095, 8191, 32767, 65535, 69999):
        ang = p * w
        ref_c = np.float32(spec.amp * np.cos(ang)).astype(np.float64)
        ref_s = np.float32(spec.amp * np.sin(ang)).astype(np.float64)
        # fp64 evaluation on both sides, one rounding to float: equal up to 1 ulp
        assert np.max(np.abs(tab[p, :, 0] - ref_c)) <= 2.0 ** -23 * 2
        assert np.max(np.abs(tab[p, :, 1] - ref_s)) <= 2.0 ** -23 * 2


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_rope_apply_matches_oracle(d):
    gu.require_gpu()
    spec = SPECS[1] if d != 512 else SPECS[3]
    B, H, T, pos0 = 2, 3, 37, 1000
    x = randn_bf16((B, H, T, d), 99 + d)
    table = gu.rope_table(d, spec, pos0 + T)
    xg = x.cuda()
    y = torch.empty_like(xg)
    gqa.gqa_rope_apply(xg, y, B, H, T, d, pos0, table, pos0 + T)
    # in place gives the same bits
    gqa.gqa_rope_apply(xg, xg, B, H, T, d, pos0, table, pos0 + T)
    assert gqa.gqa_get_device_status() == 0
    assert torch.equal(xg, y)
    w = gu.oracle_freq(d, spec)
    xf = x.to(torch.float64).numpy()
    ref = np.empty_like(xf)
    for t in range(T):
        for b in range(B):
            for h in range(H):
                ref[b, h, t] = gu.orc().rope_rotate(xf[b, h, t], pos0 + t, w, spec.amp)
    got = y.cpu().to(torch.float64).numpy()
    # one bf16 rounding of a float32 rotation: within one bf16 ulp of the exact value
    ulp = np.maximum(np.abs(ref), 1e-30) * 2.0 ** -7
    assert np.all(np.abs(got - ref) <= ulp + 1e-6)
