"""The software exp2 of the forward kernel (csrc/nc_exp2.cuh), evaluated on
the host in float32 exactly as the device evaluates it: range reduction by
the 1.5 * 2^23 add-and-subtract, a degree-3 polynomial for 2^f on
[-1/2, 1/2], and the exponent-field add.  Its error must stay far below the
bf16 rounding (2^-9) that every probability goes through afterwards."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "causal_attention_rope_nc_b300", "csrc", "nc_exp2.cuh")


def _coeffs():
    src = open(HDR).read()
    c = {int(m.group(1)): np.float32(float(m.group(2)))
         for m in re.finditer(r"EXP2_C(\d)\s*=\s*([0-9.eE+-]+)f", src)}
    assert sorted(c) == [0, 1, 2, 3]
    return c


def exp2_poly(x: np.ndarray) -> np.ndarray:
    c = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic)).astype(np.float32)
    p = (c[3] * f + c[2]).astype(np.float32)
    p = (p * f + c[1]).astype(np.float32)
    p = (p * f + c[0]).astype(np.float32)
    bits = p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-60.0, 0.0, 2_000_001, dtype=np.float64).astype(np.float32)
    got = exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.max(np.abs(got / ref - 1.0))
    assert rel < 1.0e-4, rel          # bf16 half-ulp is 2^-9 = 1.95e-3


def test_integers_are_exact_powers_of_two_up_to_the_polynomial_constant():
    # f = 0 at integers: the result is c0 * 2^n exactly
    c0 = float(_coeffs()[0])
    n = np.arange(-100, 1, dtype=np.float32)
    assert np.allclose(exp2_poly(n).astype(np.float64), c0 * np.exp2(n.astype(np.float64)), rtol=1e-7)


def test_monotone_and_positive_on_the_softmax_range():
    x = np.linspace(-40.0, 0.0, 400_001, dtype=np.float32)
    y = exp2_poly(x)
    assert np.all(y > 0)
    assert np.all(np.diff(y.astype(np.float64)) >= 0)
