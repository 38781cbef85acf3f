"""GPU parity of SwiGLU and Softmax against the oracle over the whole range of the 16-bit inputs.

The contract keeps every intermediate in FP32 (Kernscope, "Numerical contract / SwiGLU
activation" and "/ Softmax"), so a finite bf16 input whose contract result is finite must give
that result, however large its magnitude: bf16 keeps fp32's exponent range, so gate * up can
reach 1e38 and a Softmax row can have its maximum anywhere up to 3.4e38. Each case runs every
launch shape of the op (warp rows, CTA rows with and without prefetch, the wide multi-pass
kernel, the flat walk and the row kernel of SwiGLU, and the scalar kernels) and compares element
by element with the oracle: 16-bit outputs within 1 ulp and the stated gate, infinities and NaNs
where the oracle has them.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_rmsnorm_ks_gb300 as ks
from gpu_common import compare_output
from row_wise_rmsnorm_ks_gb300 import synth

pytestmark = pytest.mark.gpu

# the largest finite magnitude each input dtype holds, as a power of ten
MAX_EXP10 = {torch.bfloat16: 38.0, torch.float16: 4.8, torch.float32: 38.0}


def _log_uniform(rng, lo, hi, n):
    return np.power(10.0, rng.uniform(lo, hi, n))


def _signs(rng, n):
    return np.where(rng.random(n) < 0.5, -1.0, 1.0)


# ----------------------------------------------------------------------------------- SwiGLU

def _silu_inputs(dt, rows, d, seed):
    """Gates and ups whose product spans the dtype's range, with both gate signs.

    bf16 and fp32: positive gates log-uniform in [1e-2, 1e30], negative gates uniform in
    [-100, 0], and up chosen so |gate * up| is log-uniform in [1e18, 1e38] (so the contract's
    result stays finite, below 1e38). fp16: the same with gates up to 5e4 and -20, and products
    up to 5e4. Each row starts with fixed cases: gates around the point where
    e^-gate leaves FP32 (-87.3 .. -89, where the sigmoid is an FP32 subnormal and then 0), large
    gates with large ups, infinite gates, and products that overflow the contract's FP32 on
    purpose (the result is then inf there too)."""
    rng = np.random.default_rng(seed)
    n = rows * d
    big = MAX_EXP10[dt] > 10
    # positive gates log-uniform; negative gates uniform down to where the sigmoid is e^gate
    # below any output (a log-uniform negative gate would give mostly zeros)
    pos = _log_uniform(rng, -2, 30, n) if big else _log_uniform(rng, -3, 4.7, n)
    neg = -rng.uniform(0.0, 100.0 if big else 20.0, n)
    g = np.where(rng.random(n) < 0.5, pos, neg)
    prod = _log_uniform(rng, 18, 38, n) if big else _log_uniform(rng, -3, 4.7, n)
    up = _signs(rng, n) * np.minimum(prod / np.maximum(np.abs(g), 1e-30), 3.0e38 if big else 6.0e4)
    g = g.reshape(rows, d)
    up = up.reshape(rows, d)
    if big:
        fixed = [(10.0, 2e18), (-60.0, 3e37), (-87.0, 3e38), (-87.5, 1e38), (-88.0, 3e38),
                 (-88.5, 3e38), (-89.0, 3e38), (-100.0, 3e38), (1e30, 1e8), (-1e30, 1e9),
                 (3e38, 0.5), (-3e38, 0.5), (1e30, 1e9), (3e38, 2.0), (40.0, -3e37),
                 (float("inf"), 1.0), (float("-inf"), 1.0), (2.0, float("inf"))]
    else:
        fixed = [(-11.0, 65504.0), (-15.0, 65504.0), (-17.0, 65504.0), (-25.0, 65504.0),
                 (65504.0, 1.0), (-65504.0, 1.0), (300.0, 300.0), (60000.0, 2.0),
                 (float("inf"), 1.0), (float("-inf"), 1.0)]
    for r in range(rows):
        for j, (a, b) in enumerate(fixed[: d]):
            g[r, (j + r) % d] = a
            up[r, (j + r) % d] = b
    x = np.concatenate([g, up], axis=1).astype(np.float32)
    # torch's cast keeps infinities (the input recipe's fp16 saturation is not wanted here)
    return torch.from_numpy(x).to(dt)


# (rows, d): the flat walk (narrow rows), the row kernel with its fitted block (16-bit rows of
# 160 and >= 448 vectors), few rows, and an odd width (scalar kernel)
SILU_SHAPES = [(700, 512), (300, 1280), (150, 3584), (40, 8192), (3, 4096), (257, 1001)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,d", SILU_SHAPES)
def test_silu_and_mul_full_range(cuda_device, dtype, rows, d):
    dt = synth.dtype_of(dtype)
    x = _silu_inputs(dt, rows, d, 901 + d)
    y = ks.silu_and_mul(x.to(cuda_device)).cpu()
    ref, _ = oracle.silu_and_mul(x)
    assert torch.equal(torch.isinf(y), torch.isinf(ref))
    # fp32 bound (8+4)*2^-24: expf within 2 ulp plus three roundings
    compare_output(y, ref, dt, 8, f"silu_and_mul full range {dtype} [{rows},{d}]")
    if dt == torch.bfloat16:
        # the contract's result is finite and nonzero for the finite-product cases
        assert torch.isfinite(ref[:, 1:]).float().mean() > 0.8


def test_silu_and_mul_overflow_cases_named(cuda_device):
    """The cases that overflowed before the sigmoid was scaled back first, one by one."""
    g = [10.0, -60.0, -87.5, -88.5, 1e30]
    up = [2e18, 3e37, 1e38, 3e38, 1e8]
    x = torch.tensor([g + up], dtype=torch.float32).to(torch.bfloat16)
    y = ks.silu_and_mul(x.to(cuda_device)).cpu()
    ref, _ = oracle.silu_and_mul(x)
    assert torch.isfinite(ref).all() and torch.isfinite(y).all()
    compare_output(y, ref, torch.bfloat16, 8, "silu_and_mul named overflow cases")


# ----------------------------------------------------------------------------------- Softmax

def _softmax_inputs(dt, rows, h, seed):
    """Rows whose maximum spans the dtype's range, positive and negative, with ties at the
    maximum, moderate rows whose outputs are not one-hot at the dtype's spacing, and rows with
    NaN, +inf, -inf masks and all -inf mixed in."""
    rng = np.random.default_rng(seed)
    top = MAX_EXP10[dt]
    lo = 6.0 if top > 10 else 2.0
    x = np.empty((rows, h), dtype=np.float64)
    kinds = 9
    for r in range(rows):
        k = r % kinds
        m = 10.0 ** rng.uniform(lo, top - 0.05)
        u = rng.uniform(-1.0, 1.0, h)
        if k in (0, 3, 4, 5):      # large positive maximum, ties at it
            x[r] = m * u
            x[r, rng.integers(0, h, 3)] = m
        elif k == 1:               # large negative maximum
            x[r] = -m * (1.0 + np.abs(u))
            x[r, rng.integers(0, h)] = -m
        elif k == 2:               # moderate: spacing of the dtype near c gives non-trivial exps
            c = 10.0 ** rng.uniform(1.0, 3.0 if top > 10 else 3.5)
            x[r] = c * np.sign(u[0]) + rng.standard_normal(h) * 4.0
        elif k == 6:               # all -inf
            x[r] = -np.inf
        elif k == 7:               # one huge constant: uniform outputs
            x[r] = m
        else:                      # one huge negative constant: uniform outputs
            x[r] = -m
        if k == 3:
            x[r, rng.integers(0, h, 2)] = -np.inf   # masked entries
        if k == 4:
            x[r, rng.integers(0, h)] = np.nan
        if k == 5:
            x[r, rng.integers(0, h)] = np.inf
    return torch.from_numpy(x.astype(np.float32)).to(dt)


# (rows, h): warp rows (many narrow rows), CTA rows without prefetch (128..1024 vectors), with
# prefetch (1025..2048 vectors), the wide multi-pass kernel (> 2048 vectors), few rows, and
# widths that are not a whole number of 16-byte vectors (scalar kernel)
SOFTMAX_SHAPES = [(1001, 16), (1001, 512), (400, 4096), (200, 12288), (40, 20480), (7, 8192),
                  (300, 7), (50, 1001)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,h", SOFTMAX_SHAPES)
def test_softmax_full_range(cuda_device, dtype, rows, h):
    dt = synth.dtype_of(dtype)
    x = _softmax_inputs(dt, rows, h, 951 + h)
    y = ks.softmax(x.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(x)
    assert torch.equal(torch.isnan(y), torch.isnan(ref))
    nan_rows = torch.isnan(ref).any(dim=1)
    assert bool(torch.isnan(ref[nan_rows]).all())
    compare_output(y[~nan_rows], ref[~nan_rows], dt, h, f"softmax full range {dtype} [{rows},{h}]")
    # a NaN-free row sums to about 1 (the one-hot rows exactly)
    s = ref[~nan_rows].double().sum(dim=1)
    assert bool(((s - 1.0).abs() < 0.02 * max(1, h // 512)).all())


def test_softmax_large_maximum_named(cuda_device):
    """The row that came out NaN when -max * log2(e) was folded into one rounded FP32 bias."""
    x = torch.tensor([[3e9, 3e9 * (1 - 1e-6), 3e9 - 1, 1.5e9]] * 3, dtype=torch.float32)
    x[1] *= -1.0
    x[2] *= 1e29
    xb = x.to(torch.bfloat16)
    y = ks.softmax(xb.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(xb)
    assert not torch.isnan(ref).any() and not torch.isnan(y).any()
    compare_output(y, ref, torch.bfloat16, 4, "softmax named large maximum")
