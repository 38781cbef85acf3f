"""Pins for the oracle's hand-written casts (Kernscope "Numerical contract": cast_to_input_dtype,
read as IEEE round-to-nearest-even).

Decoding is checked over all 2^16 encodings against torch's own decoding; encoding against
torch's float->bf16/fp16 casts on random, tie and range-edge values, and against exact integer
rounding of rationals for doubles that are not fp32 values.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from helpers import FORMATS, bits_equal, exact_round

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_all_encodings(dtype):
    bits = torch.arange(-(1 << 15), 1 << 15, dtype=torch.int32).to(torch.int16)
    t = bits.view(dtype)
    ours = oracle.decode(t)
    ref = t.to(torch.float64)
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(ours), nan)
    assert torch.equal(ours[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert torch.equal(torch.signbit(ours[~nan]), torch.signbit(ref[~nan]))


def _fp32_probe_values(seed=7):
    rng = np.random.default_rng(seed)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e4).astype(np.float32),
        (rng.standard_normal(20000) * 1e-6).astype(np.float32),       # fp16 subnormal range
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),       # fp32 subnormals
        (rng.uniform(6.0e4, 7.0e4, 5000) * rng.choice([-1, 1], 5000)).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.996, 65520.0, 3.3895e38,
                  3.4028235e38, 1.0e-45, 5.96e-8, 2.98e-8, 2.9802322e-08], dtype=np.float32),
        # raw random bit patterns over the whole fp32 range (NaNs removed below)
        rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    v = np.concatenate(parts)
    return torch.from_numpy(v[~np.isnan(v)])


def _ties(dtype):
    """fp32 values exactly halfway between neighbouring dtype values (plus one ulp either side),
    where round-half-even decides."""
    bits = torch.arange(0, 0x7F00 if dtype == torch.bfloat16 else 0x7BFF, 37,
                        dtype=torch.int32).to(torch.int16)
    lo = bits.view(dtype).float()
    hi = (bits + 1).view(dtype).float()
    mid = ((lo.double() + hi.double()) / 2).float()  # exact in fp32 for 16-bit neighbours
    up = torch.nextafter(mid, torch.tensor(float("inf")))
    dn = torch.nextafter(mid, torch.tensor(float("-inf")))
    v = torch.cat([mid, up, dn])
    return torch.cat([v, -v])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_encode_matches_torch_cast(dtype):
    v = torch.cat([_fp32_probe_values(), _ties(dtype)])
    ours = oracle.encode(v.double(), dtype)
    ref = v.to(dtype)
    assert bits_equal(ours, ref)


def test_encode_fp32_identity_and_nan():
    v = _fp32_probe_values()
    assert bits_equal(oracle.encode(v.double(), torch.float32), v)
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        out = oracle.encode(torch.tensor([float("nan")], dtype=torch.float64), dt)
        assert torch.isnan(out.float()).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_encode_from_double_matches_exact_rounding(dtype):
    """Doubles that are not fp32 values must round once, directly (the float64 twin's final
    rounding), not through fp32."""
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(3000), rng.standard_normal(1000) * 3e4,
                        rng.standard_normal(1000) * 1e-5])
    ours = oracle.encode(torch.from_numpy(v), dtype).double()
    p, emin, emax = FORMATS[dtype]
    for got, x in zip(ours.tolist(), v.tolist()):
        ref = exact_round(Fraction(x), p, emin, emax)
        assert Fraction(got) == ref if not isinstance(ref, float) else got == ref, (x, got, ref)
