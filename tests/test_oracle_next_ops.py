"""Pins for the oracle's SwiGLU, Softmax and LayerNorm (Kernscope, "Numerical contract": SwiGLU
activation, Softmax; LayerNorm is only named on kernel-set's operator list and is read as the
standard definition with FP32 steps).

Each is fixed by something other than the oracle: a 60-digit decimal brute force, closed forms,
invariants, the contracts' stated non-finite rules, and torch's own fp32 routines.
"""
import decimal
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import FORMATS, bits_equal, exact_round, tol_for, ulp_dist, within_tol
from row_wise_rmsnorm_ks_gb300 import synth
from fractions import Fraction

DTYPES = [torch.bfloat16, torch.float16, torch.float32]
CTX = decimal.Context(prec=60)


def D(v):
    return CTX.create_decimal_from_float(float(v))


def round_like(values, dtype):
    p, emin, emax = FORMATS[dtype]
    return torch.tensor([float(exact_round(Fraction(v), p, emin, emax)) for v in values],
                        dtype=torch.float64).to(dtype)


def rel_err(u, exact):
    ex = torch.tensor(exact, dtype=torch.float64)
    return ((u.double() - ex).abs() / ex.abs().clamp_min(1e-30)).max().item()


# ----------------------------------------------------------------------------------- SwiGLU

def exact_swiglu(g, up):
    g, up = D(g), D(up)
    sig = CTX.divide(1, CTX.add(1, CTX.exp(CTX.minus(g))))
    return float(CTX.multiply(CTX.multiply(g, sig), up))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("d", [1, 5, 64, 1000])
def test_swiglu_vs_exact(dtype, d):
    x = synth.cast(synth.normal_np((4, 2 * d), 500 + d, std=3.0), dtype)
    out, u = oracle.silu_and_mul(x)
    assert out.shape == (4, d)
    for i in range(4):
        g, up = x[i, :d].double().tolist(), x[i, d:].double().tolist()
        ex = [exact_swiglu(a, b) for a, b in zip(g, up)]
        if dtype != torch.float32:
            assert int(ulp_dist(out[i], round_like(ex, dtype)).max()) <= 1
        # exp correctly rounded, then 1+e, 1/den, g*sig, *up: a few fp32 roundings
        assert rel_err(u[i], ex) <= 6 * 2.0 ** -24


def test_swiglu_closed_forms_and_extremes():
    g = torch.tensor([[0.0, 30.0, -30.0, 100.0, -100.0, float("inf"), float("-inf"), 2.0]])
    up = torch.tensor([[7.0, 3.0, 5.0, -2.0, 4.0, 1.0, 1.0, 0.0]])
    x = torch.cat([g, up], dim=1)
    out, _ = oracle.silu_and_mul(x)
    o = out[0].tolist()
    assert o[0] == 0.0                                  # g = 0: sigmoid(0) = 1/2, 0 * 1/2 = 0
    assert o[1] == 90.0                                 # sigmoid(30) rounds to 1 in fp32
    assert abs(o[2]) < 1e-10 and o[2] < 0               # -30 * e^-30 * 5, tiny and negative
    assert o[3] == -200.0
    assert o[4] == 0.0                                  # e^100 overflows fp32: sigmoid = 0
    assert o[5] == float("inf")                         # +inf * 1 * 1
    assert math.isnan(o[6])                             # -inf * sigmoid(-inf) = -inf * 0
    assert o[7] == 0.0                                  # up = 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(8, 2 * 4096), (3, 2 * 7), (0, 2 * 16), (2, 3, 2 * 5)])
def test_swiglu_vs_torch(dtype, shape):
    """Kernscope's checks: odd D, empty batches, leading dimensions; torch's fp32 silu."""
    x = synth.cast(synth.normal_np(shape, 7), dtype)
    d = shape[-1] // 2
    out, _ = oracle.silu_and_mul(x)
    ref = (F.silu(x[..., :d].float()) * x[..., d:].float()).to(dtype)
    assert out.shape == ref.shape
    if out.numel():
        assert int(ulp_dist(out, ref).max()) <= 1


# ----------------------------------------------------------------------------------- Softmax

def exact_softmax(row):
    m = max(row)
    ex = [CTX.exp(CTX.subtract(D(v), D(m))) for v in row]
    s = sum(ex, decimal.Decimal(0))
    return [float(CTX.divide(e, s)) for e in ex]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [1, 2, 5, 17, 1000, 4096])
def test_softmax_vs_exact(dtype, H):
    x = synth.cast(synth.normal_np((3, H), 600 + H, std=4.0), dtype)
    out, u = oracle.softmax(x)
    for i in range(3):
        ex = exact_softmax(x[i].double().tolist())
        if dtype != torch.float32:
            assert int(ulp_dist(out[i], round_like(ex, dtype)).max()) <= 1
        # the fp32 sum of H positive terms: relative error about H * 2^-24, plus a few roundings
        assert rel_err(u[i], ex) <= (H + 8) * 2.0 ** -24


def test_softmax_wide_fp16_denominator():
    """Kernscope's 65536-column FP16 case checks FP32 denominator accumulation."""
    x = synth.cast(synth.normal_np((1, 65536), 61), torch.float16)
    out, u = oracle.softmax(x)
    ex = exact_softmax(x[0].double().tolist())
    assert int(ulp_dist(out[0], round_like(ex, torch.float16)).max()) <= 1
    assert abs(float(u[0].double().sum()) - 1.0) < 1e-3


@pytest.mark.parametrize("H", [1, 4, 7, 64, 1000])
def test_softmax_uniform_row(H):
    x = torch.full((2, H), 3.5, dtype=torch.float32)
    out, _ = oracle.softmax(x)
    want = float(np.float32(1.0) / np.float32(H))   # exp(0) = 1, sum = H exactly
    assert (out == want).all()


def test_softmax_shift_invariance():
    x = torch.tensor(np.random.default_rng(3).integers(-20, 20, (4, 300)), dtype=torch.float32)
    a, _ = oracle.softmax(x)
    b, _ = oracle.softmax(x + 8.0)                  # exact shift: z = x - max is unchanged
    assert bits_equal(a, b)


def test_softmax_nonfinite_rules():
    """Kernscope: -inf masks entries of a row with finite values; rows with NaN or +inf, and rows
    all -inf, produce NaN."""
    inf, nan = float("inf"), float("nan")
    x = torch.tensor([[1.0, -inf, 2.0, -inf],
                      [1.0, nan, 2.0, 3.0],
                      [1.0, inf, 2.0, 3.0],
                      [-inf, -inf, -inf, -inf],
                      [0.5, 0.25, -inf, 1.0]], dtype=torch.float32)
    out, _ = oracle.softmax(x)
    assert out[0, 1] == 0 and out[0, 3] == 0
    ref0, _ = oracle.softmax(torch.tensor([[1.0, 2.0]]))
    assert out[0, 0] == ref0[0, 0] and out[0, 2] == ref0[0, 1]
    for r in (1, 2, 3):
        assert torch.isnan(out[r]).all()
    assert out[4, 2] == 0 and torch.isfinite(out[4]).all()
    ref = torch.softmax(x, dim=-1)
    assert torch.equal(torch.isnan(out), torch.isnan(ref))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(2, 5), (512, 1024), (4, 16384), (0, 8)])
def test_softmax_vs_torch(dtype, shape):
    x = synth.cast(synth.normal_np(shape, 9, std=3.0), dtype)
    out, _ = oracle.softmax(x)
    ref = torch.softmax(x.float(), dim=-1).to(dtype)
    if out.numel():
        assert int(ulp_dist(out, ref).max()) <= 1


# --------------------------------------------------------------------------------- LayerNorm

def exact_layer_norm(row, w, b, eps):
    xs = [D(v) for v in row]
    H = len(xs)
    mean = CTX.divide(sum(xs, decimal.Decimal(0)), H)
    var = CTX.divide(sum((CTX.multiply(v - mean, v - mean) for v in xs), decimal.Decimal(0)), H)
    rstd = CTX.divide(1, CTX.sqrt(CTX.add(var, D(eps))))
    return [float(CTX.add(CTX.multiply(CTX.multiply(v - mean, rstd), D(wj)), D(bj)))
            for v, wj, bj in zip(xs, w, b)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [2, 3, 17, 1000, 4096])
def test_layer_norm_vs_exact(dtype, H):
    x = synth.cast(synth.normal_np((3, H), 700 + H) + np.float32(0.5), dtype)
    w = synth.weight(H, dtype, seed=701)
    b = synth.cast(synth.normal_np((H,), 702, std=0.1), dtype)
    eps = 1e-5
    eps32 = float(np.float32(eps))
    out, u = oracle.layer_norm(x, w, b, eps)
    for i in range(3):
        ex = exact_layer_norm(x[i].double().tolist(), w.double().tolist(), b.double().tolist(),
                              eps32)
        if dtype != torch.float32:
            # the bias is added last and can cancel: 1 ulp away from 0, the tolerance gate near it
            ref = round_like(ex, dtype)
            away = ref.double().abs() > 0.05
            assert int(ulp_dist(out[i][away], ref[away]).max()) <= 1
            rtol, atol = tol_for(dtype, H)
            assert within_tol(out[i], ref, rtol, atol)[0]
        # two fp32 sums and a few roundings; bias added last can cancel, so an absolute floor
        exact_t = torch.tensor(ex, dtype=torch.float64)
        err = (u[i].double() - exact_t).abs()
        assert bool((err <= (H + 8) * 2.0 ** -24 * (exact_t.abs() + 4.0)).all())


def test_layer_norm_constant_row_gives_bias():
    H = 64
    x = torch.full((2, H), 0.75, dtype=torch.bfloat16)
    w = synth.weight(H, torch.bfloat16)
    b = synth.cast(synth.normal_np((H,), 3), torch.bfloat16)
    out, _ = oracle.layer_norm(x, w, b, 1e-5)
    assert torch.equal(out[0].float(), b.float()) and torch.equal(out[1].float(), b.float())


def test_layer_norm_invariants_and_defaults():
    H = 4096
    x = synth.cast(synth.normal_np((8, H), 5, std=3.0), torch.float32)
    out, u = oracle.layer_norm(x, None, None, 1e-12)
    assert (u.double().mean(dim=1).abs() < 1e-5).all()
    assert ((u.double().pow(2).mean(dim=1) - 1).abs() < 1e-4).all()
    ones, zeros = torch.ones(H), torch.zeros(H)
    out2, _ = oracle.layer_norm(x, ones, zeros, 1e-12)
    assert bits_equal(out, out2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(5,), (2, 3, 5), (3, 1000), (128, 4096)])
def test_layer_norm_vs_torch(dtype, shape):
    H = shape[-1]
    x = synth.cast(synth.normal_np(shape, 11), dtype)
    w = synth.weight(H, dtype)
    b = synth.cast(synth.normal_np((H,), 12, std=0.1), dtype)
    out, _ = oracle.layer_norm(x, w, b, 1e-5)
    ref = F.layer_norm(x.float(), (H,), w.float(), b.float(), 1e-5).to(dtype)
    away = ref.double().abs() > 0.05
    assert int(ulp_dist(out[away], ref[away]).max()) <= 1
    rtol, atol = tol_for(dtype, H)
    assert within_tol(out, ref, rtol, atol)[0]
