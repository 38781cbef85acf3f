"""Shared test helpers: ulp distances, the output tolerance gate, exact high-precision RMSNorm.

Nothing here imports the CUDA binding or the oracle; the exact reference below is written with
Python's decimal module, independently of both.
"""
from __future__ import annotations

import decimal
from fractions import Fraction

import torch

# Output tolerance gate (|d| <= rtol*|ref| + atol), from the stated contract tolerance: bf16
# 1e-2/1e-3, fp16 2e-3/1e-4. fp32 is not a graded dtype; its bound is derived from the
# arithmetic: the oracle sums squares left to right, whose relative error is at most about
# H*2^-24; the scale inherits half of it and the two products add two rounding errors.
TOL = {torch.bfloat16: (1e-2, 1e-3), torch.float16: (2e-3, 1e-4)}


def fp32_tol(hidden: int):
    return (hidden * 2.0 ** -24 + 4 * 2.0 ** -24, 1e-30)


def tol_for(dtype, hidden: int):
    return TOL.get(dtype) or fp32_tol(hidden)


def _ordered(t: torch.Tensor) -> torch.Tensor:
    """Map float bit patterns to integers that are monotone in value (for ulp distances)."""
    if t.dtype in (torch.bfloat16, torch.float16):
        i = t.contiguous().view(torch.int16).to(torch.int64)
        sign_mask = 0x8000
        mag = i & 0x7FFF
    else:
        i = t.contiguous().view(torch.int32).to(torch.int64)
        sign_mask = 0x80000000
        mag = i & 0x7FFFFFFF
    neg = (i & sign_mask) != 0
    return torch.where(neg, -mag, mag)


def ulp_dist(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """ulp distance between two same-dtype tensors (+0 and -0 are 0 apart). NaN pairs count 0
    only when both are NaN; a NaN against a number counts as a huge distance."""
    assert a.dtype == b.dtype and a.shape == b.shape
    d = (_ordered(a) - _ordered(b)).abs()
    na, nb = torch.isnan(a.float()), torch.isnan(b.float())
    d = torch.where(na & nb, torch.zeros_like(d), d)
    d = torch.where(na ^ nb, torch.full_like(d, 1 << 40), d)
    return d


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality, with any NaN equal to any NaN."""
    if a.dtype != b.dtype or a.shape != b.shape:
        return False
    ia = a.contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32)
    na, nb = torch.isnan(a.float()), torch.isnan(b.float())
    same = (ia == ib) | (na & nb)
    return bool(same.all())


def within_tol(out: torch.Tensor, ref: torch.Tensor, rtol: float, atol: float):
    """Element-wise |out - ref| <= rtol*|ref| + atol in float64; NaN must meet NaN and inf must
    meet the same inf. Returns (ok, worst excess, index of worst)."""
    o, r = out.double(), ref.double()
    nan_ok = torch.isnan(o) == torch.isnan(r)
    inf_ok = torch.where(torch.isinf(r) | torch.isinf(o), o == r, torch.ones_like(nan_ok))
    fin = torch.isfinite(o) & torch.isfinite(r)
    err = torch.where(fin, (o - r).abs() - (rtol * r.abs() + atol), torch.zeros_like(o))
    ok = bool(nan_ok.all()) and bool(inf_ok.all()) and bool((err <= 0).all())
    worst = float(err.max()) if err.numel() else 0.0
    idx = int(err.argmax()) if err.numel() else -1
    return ok, worst, idx


# ------------------------------------------------------------------ exact RMSNorm (decimal)

_CTX = decimal.Context(prec=80)


def _dec(v: float) -> decimal.Decimal:
    return _CTX.create_decimal_from_float(float(v))  # exact: binary floats are finite decimals


def exact_rms_norm_row(x_vals, w_vals, eps: float):
    """Exact-to-80-digits RMSNorm of one row from its float values (decoded inputs):
    y_j = x_j * w_j / sqrt(sum(x^2)/H + eps). Returns Python floats (correctly rounded)."""
    H = len(x_vals)
    xs = [_dec(v) for v in x_vals]
    ss = sum((_CTX.multiply(a, a) for a in xs), decimal.Decimal(0))
    mean = _CTX.divide(ss, decimal.Decimal(H))
    root = _CTX.sqrt(_CTX.add(mean, _dec(eps)))
    return [float(_CTX.divide(_CTX.multiply(a, _dec(w)), root)) for a, w in zip(xs, w_vals)]


def exact_fused_row(x_vals, r_vals, w_vals, eps: float):
    """Exact fused op on one row: s = x + r exactly, y = s*w/sqrt(mean(s^2)+eps).
    Returns (y floats, s floats)."""
    s = [_CTX.add(_dec(a), _dec(b)) for a, b in zip(x_vals, r_vals)]
    H = len(s)
    ss = sum((_CTX.multiply(a, a) for a in s), decimal.Decimal(0))
    root = _CTX.sqrt(_CTX.add(_CTX.divide(ss, decimal.Decimal(H)), _dec(eps)))
    y = [float(_CTX.divide(_CTX.multiply(a, _dec(w)), root)) for a, w in zip(s, w_vals)]
    return y, [float(a) for a in s]


def exact_round(value: Fraction, p: int, emin: int, emax: int) -> Fraction:
    """Round an exact rational to the nearest value with p significand bits (ties to even),
    by integer arithmetic only. Returns a Fraction, or +-inf as float on overflow."""
    if value == 0:
        return Fraction(0)
    sign = -1 if value < 0 else 1
    a = abs(value)
    # exponent of the leading bit: 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    q = Fraction(2) ** (e - (p - 1))
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * q
    max_finite = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if r > max_finite:
        return sign * float("inf")
    return sign * r


FORMATS = {torch.bfloat16: (8, -126, 127), torch.float16: (11, -14, 15),
           torch.float32: (24, -126, 127)}
