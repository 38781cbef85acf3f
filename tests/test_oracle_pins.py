"""Pins for the oracle's RMSNorm and fused residual-add RMSNorm (Kernscope "Numerical contract").

Each pin is fixed by something other than the oracle itself:
  * closed forms: a constant row c gives c*w/sqrt(c^2+eps); a zero row gives 0;
  * invariants: scaling x by a power of two leaves the unit-weight output unchanged (up to the
    eps term), the unit-weight output has RMS about 1, the stored residual is the rounded sum,
    the fused op with a zero residual is plain RMSNorm;
  * an exact (80-digit decimal) brute force on tiny and medium rows, which the oracle's final
    output must meet within 1 ulp and its pre-cast fp32 value within the fp32 error bound;
  * a library routine: torch.nn.functional.rms_norm on fp32 CPU, the same contract.
Planted mistakes each of these catches: a dropped or misplaced eps (closed form, large eps), a
wrong divisor (closed form is H-free, the brute force is not), a transposed or shifted weight
(brute force with random weight), a sign or index slip (brute force), normalising the rounded
residual sum instead of the fp32 one (pre-cast value vs the exact sum, fp16/bf16).
"""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import (FORMATS, bits_equal, exact_fused_row, exact_rms_norm_row, exact_round,
                     tol_for, ulp_dist, within_tol)
from row_wise_rmsnorm_ks_gb300 import synth

DTYPES = [torch.bfloat16, torch.float16, torch.float32]


def _round_like(values, dtype):
    p, emin, emax = FORMATS[dtype]
    out = []
    for v in values:
        r = exact_round(Fraction(v), p, emin, emax)
        out.append(float(r))
    return torch.tensor(out, dtype=torch.float64).to(dtype)


# ----------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("c", [1.0, 0.75, -3.0, 0.3125, 1000.0])
@pytest.mark.parametrize("H", [1, 3, 1000, 4096])
@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_constant_row_closed_form(dtype, c, H, eps):
    x = torch.full((2, H), c, dtype=dtype)
    w = synth.weight(H, dtype)
    y, u = oracle.rms_norm(x, w, eps)
    eps32 = float(np.float32(eps))
    cd = float(x[0, 0].double())
    denom = math.sqrt(cd * cd + eps32)
    exact = [cd * float(wj) / denom for wj in w.double().tolist()]
    ref = _round_like(exact, dtype)
    if dtype != torch.float32:  # fp32 output is u itself, bounded below
        assert int(ulp_dist(y[0], ref).max()) <= 1
    # the fp32 value before the cast: a few fp32 ulps (sum of H equal squares is exact up to
    # H*2^-24 relative in fp32; the rest is three roundings)
    rel = ((u[0].double() - torch.tensor(exact)).abs() / torch.tensor(exact).abs()).max()
    assert float(rel) <= (H + 8) * 2.0 ** -24


@pytest.mark.parametrize("dtype", DTYPES)
def test_zero_row_is_zero(dtype):
    x = torch.zeros((3, 257), dtype=dtype)
    w = synth.weight(257, dtype)
    y, _ = oracle.rms_norm(x, w, 1e-6)
    assert (y.double() == 0).all()
    xf, rf, _ = oracle.fused_add_rms_norm(x, torch.zeros_like(x), w, 1e-6)
    assert (xf.double() == 0).all() and (rf.double() == 0).all()


# ------------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("k", [-3, 4])
def test_scale_invariance_unit_weight(dtype, k):
    x = synth.cast(synth.normal_np((16, 777), 5), dtype)
    w = torch.ones(777, dtype=dtype)
    xs = (x.double() * 2.0 ** k).to(dtype)
    if not torch.equal(xs.double() * 2.0 ** -k, x.double()):
        pytest.skip("scaling is not exact in this dtype (fp16 subnormals)")
    y1, _ = oracle.rms_norm(x, w, 1e-12)
    y2, _ = oracle.rms_norm(xs, w, 1e-12)
    assert int(ulp_dist(y1, y2).max()) <= 1


@pytest.mark.parametrize("dtype", DTYPES)
def test_unit_weight_rms_is_one(dtype):
    x = synth.cast(synth.normal_np((32, 4096), 9, std=3.0), dtype)
    w = torch.ones(4096, dtype=dtype)
    y, u = oracle.rms_norm(x, w, 1e-6)
    rms_u = u.double().pow(2).mean(dim=1).sqrt()
    assert ((rms_u - 1).abs() < 1e-5).all()
    rms_y = y.double().pow(2).mean(dim=1).sqrt()
    assert ((rms_y - 1).abs() < 5e-3).all()


@pytest.mark.parametrize("dtype", DTYPES)
def test_residual_is_rounded_fp32_sum(dtype):
    x = synth.cast(synth.normal_np((64, 1000), 1), dtype)
    r = synth.cast(synth.normal_np((64, 1000), 2, std=2.0), dtype)
    w = synth.weight(1000, dtype)
    _, ro, _ = oracle.fused_add_rms_norm(x, r, w, 1e-6)
    assert bits_equal(ro, (x.float() + r.float()).to(dtype))
    # numpy's fp32 add and cast agree for the fp16 case
    if dtype == torch.float16:
        ref = (x.numpy().astype(np.float32) + r.numpy().astype(np.float32)).astype(np.float16)
        assert bits_equal(ro, torch.from_numpy(ref))


@pytest.mark.parametrize("dtype", DTYPES)
def test_fused_with_zero_residual_is_plain(dtype):
    x = synth.cast(synth.normal_np((20, 1536), 4), dtype)
    w = synth.weight(1536, dtype)
    y, u = oracle.rms_norm(x, w, 1e-6)
    xf, rf, uf = oracle.fused_add_rms_norm(x, torch.zeros_like(x), w, 1e-6)
    assert bits_equal(xf, y) and bits_equal(rf, x)
    assert torch.equal(u, uf)


def test_inputs_not_modified_and_inplace_alias_semantics():
    x = synth.cast(synth.normal_np((4, 64), 4), torch.bfloat16)
    r = synth.cast(synth.normal_np((4, 64), 5), torch.bfloat16)
    w = synth.weight(64, torch.bfloat16)
    x0, r0 = x.clone(), r.clone()
    oracle.fused_add_rms_norm(x, r, w)
    assert bits_equal(x, x0) and bits_equal(r, r0)


# ------------------------------------------------------- exact brute force on tiny/medium rows

def _rows(dtype, H, n, seed, heavy=False):
    a = synth.student_t3_np((n, H), seed) if heavy else synth.normal_np((n, H), seed)
    if heavy:
        a[0] *= 1e3
    return synth.cast(a, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [1, 2, 3, 5, 8, 17, 1000])
def test_rms_norm_vs_exact(dtype, H):
    n = 6 if H < 1000 else 3
    x = _rows(dtype, H, n, 100 + H, heavy=(H == 17))
    w = synth.weight(H, dtype, seed=200 + H)
    eps = 1e-6
    y, u = oracle.rms_norm(x, w, eps)
    yd = oracle.rms_norm_f64(x, w, eps)
    eps32 = float(np.float32(eps))
    for i in range(n):
        exact = exact_rms_norm_row(x[i].double().tolist(), w.double().tolist(), eps32)
        ex = torch.tensor(exact, dtype=torch.float64)
        if dtype != torch.float32:
            assert int(ulp_dist(y[i], _round_like(exact, dtype)).max()) <= 1
        rel = ((u[i].double() - ex).abs() / ex.abs().clamp_min(1e-300)).max()
        assert float(rel) <= (H + 8) * 2.0 ** -24, (i, float(rel))
        # the float64 twin agrees with the exact value to double precision
        relf = ((yd[i] - ex).abs() / ex.abs().clamp_min(1e-300)).max()
        assert float(relf) <= (H + 8) * 2.0 ** -52


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H", [1, 2, 3, 5, 8, 17, 1000])
def test_fused_vs_exact(dtype, H):
    n = 6 if H < 1000 else 3
    x = _rows(dtype, H, n, 300 + H, heavy=(H == 17))
    r = _rows(dtype, H, n, 400 + H)
    w = synth.weight(H, dtype, seed=500 + H)
    eps = 1e-6
    xo, ro, u = oracle.fused_add_rms_norm(x, r, w, eps)
    yd, sd = oracle.fused_add_rms_norm_f64(x, r, w, eps)
    eps32 = float(np.float32(eps))
    for i in range(n):
        y_ex, s_ex = exact_fused_row(x[i].double().tolist(), r[i].double().tolist(),
                                     w.double().tolist(), eps32)
        ex = torch.tensor(y_ex, dtype=torch.float64)
        if dtype != torch.float32:
            assert int(ulp_dist(xo[i], _round_like(y_ex, dtype)).max()) <= 1
        assert bits_equal(ro[i], _round_like(s_ex, dtype))
        # pre-cast value follows the unrounded fp32 sum: within the fp32 bound of the exact
        # value. Normalising the rounded 16-bit sum instead would miss by up to 2^-9 relative.
        rel = ((u[i].double() - ex).abs() / ex.abs().clamp_min(1e-300)).max()
        assert float(rel) <= (H + 8) * 2.0 ** -24, (i, float(rel))
        assert torch.allclose(sd[i], torch.tensor(s_ex, dtype=torch.float64), rtol=0, atol=0)


def test_fused_normalises_unrounded_sum_specifically():
    """Rows built so that the 16-bit rounding of s moves the output by a detectable amount in
    the fp32 pre-cast value: x = 1, r = 2^-9 (s = 1 + 2^-9, which bf16 rounds to 1)."""
    H = 4
    x = torch.tensor([[1.0, 1.0, 1.0, 1.0]], dtype=torch.bfloat16)
    r = torch.tensor([[2.0 ** -9, 0.0, 0.0, 0.0]], dtype=torch.bfloat16)
    w = torch.ones(H, dtype=torch.bfloat16)
    _, ro, u = oracle.fused_add_rms_norm(x, r, w, 1e-6)
    assert float(ro[0, 0]) == 1.0                    # stored residual is rounded
    s0 = 1.0 + 2.0 ** -9
    mean = (s0 * s0 + 3.0) / 4
    want = s0 / math.sqrt(mean + float(np.float32(1e-6)))
    assert abs(float(u[0, 0]) - want) <= 4 * 2.0 ** -24
    assert abs(float(u[0, 0]) - 1.0) > 1e-3          # the rounded sum would give ~1.0


# --------------------------------------------------------------------- library routine (torch)

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(5,), (2, 3, 5), (3, 1000), (128, 1024)])
def test_vs_torch_rms_norm(dtype, shape):
    """Kernscope's own test shapes. torch's fp32 rms_norm is the same contract with another
    summation order, so the outputs agree within 1 ulp."""
    H = shape[-1]
    x = synth.cast(synth.normal_np(shape, 42), dtype)
    w = synth.weight(H, dtype)
    y, u = oracle.rms_norm(x, w, 1e-6)
    ref32 = F.rms_norm(x.float(), (H,), w.float(), 1e-6)
    assert int(ulp_dist(y, ref32.to(dtype)).max()) <= 1
    rel = ((u.double() - ref32.double()).abs() / ref32.double().abs().clamp_min(1e-30)).max()
    assert float(rel) <= (H + 8) * 2.0 ** -24
    rtol, atol = tol_for(dtype, H)
    ok, worst, _ = within_tol(y, ref32.to(dtype), rtol, atol)
    assert ok, worst


def test_empty_rows():
    x = torch.zeros((0, 16), dtype=torch.bfloat16)
    w = synth.weight(16, torch.bfloat16)
    y, u = oracle.rms_norm(x, w)
    assert y.shape == (0, 16)
    xo, ro, _ = oracle.fused_add_rms_norm(x, x.clone(), w)
    assert xo.shape == (0, 16) and ro.shape == (0, 16)


def test_nonfinite_propagation():
    """IEEE propagation (the pages state no rule for RMSNorm): an inf in a row gives ss = inf,
    scale = 0, so finite elements become 0 and the inf element NaN."""
    x = torch.tensor([[1.0, float("inf"), 2.0], [1.0, float("nan"), 1.0]], dtype=torch.float32)
    w = torch.ones(3)
    y, _ = oracle.rms_norm(x, w)
    assert y[0, 0] == 0 and torch.isnan(y[0, 1]) and y[0, 2] == 0
    assert torch.isnan(y[1]).all()
