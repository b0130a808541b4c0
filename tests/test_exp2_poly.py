"""The FMA-pipe 2^x of the prefill softmax: its constants and its error bound.

The kernels carry the polynomial's coefficients as float literals; they must be the ones
that exp2_poly.py derives (Chebyshev interpolation, Cody-Waite reduction), and the fp32
evaluation, step for step as the kernel does it, must stay within the stated bound of
the exact 2^x, and give exactly 0 for -inf and 1 for 0.
"""
import re
from pathlib import Path

import numpy as np

from global_causal_gqa_gb300 import exp2_poly

HEADER = Path(__file__).resolve().parents[1] / "global_causal_gqa_gb300" / "csrc" / "ptx.cuh"


def test_header_constants_match_the_derivation():
    text = HEADER.read_text()
    lits = dict(re.findall(r"constexpr float (kExp2A\d) = ([0-9a-fx.p+-]+)f;", text))
    got = [np.float32(float.fromhex(lits[f"kExp2A{i}"])) for i in range(3)]
    assert got == list(exp2_poly.coefficients())


def test_relative_error_bound_and_special_values():
    xs = np.concatenate([np.linspace(-126.0, 8.0, 1_000_001), np.arange(-126, 9) + 0.5])
    xs = xs.astype(np.float32)
    rel = np.abs(exp2_poly.evaluate_fp32(xs).astype(np.float64) / np.exp2(xs.astype(np.float64)) - 1)
    assert rel.max() < exp2_poly.REL_ERR_BOUND
    special = exp2_poly.evaluate_fp32(np.array([-np.inf, -1000.0, -127.0, 0.0, 1.0, -1.0], np.float32))
    assert special[0] == 0.0 and special[1] == 0.0 and special[2] == 0.0
    assert special[3] == 1.0 and special[4] == 2.0 and special[5] == 0.5


def test_monotone_on_a_fine_grid():
    xs = np.linspace(-20.0, 8.0, 200_001).astype(np.float32)
    y = exp2_poly.evaluate_fp32(xs)
    assert np.all(np.diff(y.astype(np.float64)) >= -1e-7 * y[1:])
