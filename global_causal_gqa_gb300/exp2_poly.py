"""Coefficients of the FMA-pipe 2^x used by the prefill softmax kernels.

Method: Cody-Waite style range reduction, 2^x = 2^n * 2^f with n = rint(x) and
f in [-1/2, 1/2], and 2^f = 1 + f * q(f), where q is the degree-2 polynomial that
interpolates g(f) = (2^f - 1) / f at the three Chebyshev nodes of [-1/2, 1/2].
Keeping the constant term at exactly 1 makes 2^0 exact, so an input clamped to the
bottom of the range (-127, where n carries all of it and f = 0) yields +0.0 exactly.

Run as a script to print the coefficients as C float literals; the CUDA header holds
the same literals and a CPU test checks that they agree with this file and that the
relative error of the fp32 evaluation stays below ``REL_ERR_BOUND``.
"""
import numpy as np

REL_ERR_BOUND = 2.5e-4   # vs bf16's half-ulp of 2^-9 ~= 1.95e-3, applied to P right after


def coefficients():
    """(a0, a1, a2) of q(f) = a0 + a1 f + a2 f^2, rounded to float32."""
    k = np.arange(3)
    nodes = 0.5 * np.cos((2 * k + 1) * np.pi / 6)           # Chebyshev nodes on [-1/2, 1/2]
    g = np.expm1(nodes * np.log(2.0)) / nodes
    a = np.linalg.solve(np.vander(nodes, 3, increasing=True), g)
    return tuple(np.float32(c) for c in a)


def evaluate_fp32(x):
    """The kernel's arithmetic, step by step in float32 (numpy), for checking."""
    a0, a1, a2 = coefficients()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-127.0))
    magic = np.float32(12582912.0)                          # 1.5 * 2^23: add rounds to int
    t = (x + magic).astype(np.float32)
    n_f = (t - magic).astype(np.float32)
    f = (x - n_f).astype(np.float32)
    u = (a2 * f + a1).astype(np.float32)
    u = (u * f + a0).astype(np.float32)
    p = (u * f + np.float32(1.0)).astype(np.float32)
    bits = p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    for name, c in zip(("a0", "a1", "a2"), coefficients()):
        print(f"{name} = {float(c).hex()}  ({float(c):.9g}f)")
    xs = np.linspace(-60.0, 8.0, 2_000_001, dtype=np.float64).astype(np.float32)
    rel = np.abs(evaluate_fp32(xs).astype(np.float64) / np.exp2(xs.astype(np.float64)) - 1)
    print("max relative error", rel.max())
