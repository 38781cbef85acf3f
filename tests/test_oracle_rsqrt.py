"""Pins for the oracle's reciprocal square root, read as the correctly rounded fp32 value of
1/sqrt(v) (Kernscope "Numerical contract": scale = rsqrt(mean + eps), FP32 intermediates).

The reference here is exact: for adjacent floats a < b around 1/sqrt(v), 1/sqrt(v) lies above
their midpoint m exactly when m*m*v < 1, decided with Python Fractions.
"""
import math
from fractions import Fraction

import numpy as np
import torch

import oracle


def _exact_rsqrt_rn(v: float) -> float:
    f32 = np.float32
    r = f32(1.0 / math.sqrt(v))
    V = Fraction(float(v))

    def above(m):  # 1/sqrt(v) > m  <=>  m^2 v < 1
        return m * m * V < 1

    while True:
        up = np.nextafter(r, f32(np.inf))
        m = (Fraction(float(r)) + Fraction(float(up))) / 2
        if above(m):
            r = up
        else:
            break
    while True:
        dn = np.nextafter(r, f32(0))
        m = (Fraction(float(r)) + Fraction(float(dn))) / 2
        if not above(m) and m * m * V != 1:
            r = dn
        else:
            break
    return float(r)


def test_rsqrt_exact_on_wide_sample():
    rng = np.random.default_rng(3)
    mant = rng.uniform(1.0, 2.0, 3000)
    expo = rng.integers(-149, 127, 3000)
    v = np.ldexp(mant, expo).astype(np.float32)
    v = v[(v > 0) & np.isfinite(v)]
    extra = np.array([1.0, 4.0, 0.25, 2.0, 0.5, 16.0, 1e-6, 1e-5, 1.000001, 3.4028235e38,
                      1.4e-45, 1.1754944e-38, 9.0, 1.0 + 2 ** -23, 1.0 - 2 ** -24],
                     dtype=np.float32)
    v = np.concatenate([v, extra])
    ours = oracle.rsqrt(torch.from_numpy(v)).tolist()
    for vi, o in zip(v.tolist(), ours):
        assert o == _exact_rsqrt_rn(vi), vi


def test_rsqrt_perfect_squares_are_exact():
    v = torch.tensor([4.0 ** k for k in range(-60, 60)], dtype=torch.float32)
    out = oracle.rsqrt(v)
    ref = torch.tensor([2.0 ** -k for k in range(-60, 60)], dtype=torch.float32)
    assert torch.equal(out, ref)


def test_rsqrt_specials():
    v = torch.tensor([0.0, -0.0, float("inf"), float("nan"), -1.0], dtype=torch.float32)
    out = oracle.rsqrt(v)
    assert out[0] == float("inf") and out[1] == float("inf")
    assert out[2] == 0.0
    assert torch.isnan(out[3]) and torch.isnan(out[4])
