"""The polynomial exp2 used on the FMA pipe (csrc/exp2_poly.cuh) against the
mathematics: an fp32 emulation of its range reduction and Horner evaluation
stays within 3e-7 relative of 2^x (fp64) over the range the kernels feed it,
comparable to the hardware exp2 approximation's 2-ulp bound."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "attention_scored_sparse_gb300", "csrc", "exp2_poly.cuh")


def coefficients():
    txt = open(HDR).read()
    c = dict((int(k), float(v)) for k, v in re.findall(r"kExp2C(\d) = ([-0-9.e]+)f;", txt))
    return np.array([c[k] for k in sorted(c)], dtype=np.float32)


def exp2_emulated(x):
    """fp32 emulation: n = round(x) via the 1.5*2^23 shift, f = x - n,
    Horner with one rounding per fused multiply-add, exponent add."""
    c = coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    j = (x.astype(np.float64) + 12582912.0).astype(np.float32)
    n = (j.astype(np.float64) - 12582912.0).astype(np.float32)
    f = (x.astype(np.float64) - n).astype(np.float32)
    p = np.full_like(f, c[-1])
    for k in range(len(c) - 2, -1, -1):
        p = (p.astype(np.float64) * f + np.float64(c[k])).astype(np.float32)
    bits = p.view(np.int32) + (n.astype(np.int32) << 23)
    return bits.view(np.float32)


def test_exp2_poly_relative_error_bound():
    x = np.concatenate([np.linspace(-125.9, 0.0, 2_000_001), np.linspace(-1, 1, 100001)])
    got = exp2_emulated(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float32).astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 3e-7


def test_exp2_poly_exact_powers_and_reduction():
    for k in range(-120, 2):
        assert abs(exp2_emulated(np.array([float(k)]))[0] / 2.0 ** k - 1) < 3e-7
