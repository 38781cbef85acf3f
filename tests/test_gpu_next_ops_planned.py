"""Every launch variant of SwiGLU, Softmax and LayerNorm through the explicit-plan entry points
(ks_*_planned, the C ABI), against the oracle element by element: 16-bit outputs within 1 ulp and
the stated gate, fp32 within its derived bound; LayerNorm by the same rule as its other tests
(1 ulp away from zero, the gate near it, where the bias cancels). Shapes are ragged (rows not a
multiple of a CTA's warp rows, widths not a multiple of a team's vectors).
"""
import pytest
import torch

import oracle
from gpu_common import compare_output
from helpers import tol_for, ulp_dist, within_tol
from row_wise_rmsnorm_ks_gb300 import _abi as A
from row_wise_rmsnorm_ks_gb300 import synth

pytestmark = pytest.mark.gpu
CODES = {torch.bfloat16: A.KS_DTYPE_BF16, torch.float16: A.KS_DTYPE_F16,
         torch.float32: A.KS_DTYPE_F32}
NP = A.KS_PLAN_NO_PREFETCH


def _up32(n):
    return -(-n // 32) * 32


def _vectors(dt, hidden):
    return hidden * (4 if dt == torch.float32 else 2) // 16


# Softmax / LayerNorm variants: (name, kernel, vectors per thread, block or None for "fitted",
# flags, stages[, lanes per row for warp rows])
ROW_VARIANTS = [
    ("t8v2", A.KS_KERNEL_WARP_ROW, 2, 128, 0, 0, 8), ("t8v4n", A.KS_KERNEL_WARP_ROW, 4, 96, NP, 0, 8),
    ("t16v2n", A.KS_KERNEL_WARP_ROW, 2, 64, NP, 0, 16), ("t16v4", A.KS_KERNEL_WARP_ROW, 4, 128, 0, 0, 16),
    ("w2", A.KS_KERNEL_WARP_ROW, 2, 128, 0, 0), ("w2n", A.KS_KERNEL_WARP_ROW, 2, 64, NP, 0),
    ("w4", A.KS_KERNEL_WARP_ROW, 4, 128, 0, 0), ("w4n", A.KS_KERNEL_WARP_ROW, 4, 96, NP, 0),
    ("w6", A.KS_KERNEL_WARP_ROW, 6, 128, 0, 0), ("w8n", A.KS_KERNEL_WARP_ROW, 8, 128, NP, 0),
    ("w8", A.KS_KERNEL_WARP_ROW, 8, 32, 0, 0),
    ("c1", A.KS_KERNEL_CTA_ROW, 1, None, 0, 0), ("c2", A.KS_KERNEL_CTA_ROW, 2, None, 0, 0),
    ("c4", A.KS_KERNEL_CTA_ROW, 4, None, 0, 0), ("c4n", A.KS_KERNEL_CTA_ROW, 4, None, NP, 0),
    ("ring2", A.KS_KERNEL_BULK_ROW, 4, None, 0, 2), ("ring5", A.KS_KERNEL_BULK_ROW, 4, None, 0, 5),
    ("ring2a", A.KS_KERNEL_BULK_ROW, 4, None, A.KS_PLAN_AFFINE_SMEM, 2),
    ("ring4a", A.KS_KERNEL_BULK_ROW, 4, None, A.KS_PLAN_AFFINE_SMEM, 4),
    ("wide128", A.KS_KERNEL_TWOPASS_ROW, 4, 128, 0, 0),
    ("wide512", A.KS_KERNEL_TWOPASS_ROW, 4, 512, 0, 0),
    ("wide1024", A.KS_KERNEL_TWOPASS_ROW, 4, 1024, 0, 0),
    ("scalar", A.KS_KERNEL_SCALAR, 0, 256, 0, 0),
]


def _row_plan(variant, op, dt, hidden):
    name, kernel, v, block, flags, stages = variant[:6]
    team = variant[6] if len(variant) > 6 else 32
    hv = _vectors(dt, hidden)
    if kernel != A.KS_KERNEL_SCALAR and (hidden * (4 if dt == torch.float32 else 2)) % 16:
        return None
    if kernel == A.KS_KERNEL_WARP_ROW and team * v < hv:
        return None
    if block is None:
        block = max(32, _up32(-(-hv // v)))
        # up to 1024 threads for the ring with the weight and bias in shared memory
        if block > (1024 if flags & A.KS_PLAN_AFFINE_SMEM else 512):
            return None
    if op == "layer_norm" and flags & NP:
        return None  # LayerNorm always prefetches
    affine_rows = 2 if flags & A.KS_PLAN_AFFINE_SMEM else 0
    if kernel == A.KS_KERNEL_BULK_ROW and (op != "layer_norm" or
                                           128 + (stages + affine_rows) * hv * 16 > 226 * 1024):
        return None
    if kernel == A.KS_KERNEL_TWOPASS_ROW and op == "layer_norm" and block > 512:
        return None
    return A.make_plan(kernel, v, block, stages, flags=flags, team=team)


# ragged row counts (not a multiple of a CTA's teams, so some teams of a warp have no row), widths
# of 8..64 vectors for the sub-warp teams, wider ones for the rest
SHAPES = [(333, 512), (1001, 1000), (77, 2056), (45, 4096), (9, 20480), (1003, 64), (7, 128),
          (517, 248), (2001, 256)]


@pytest.mark.parametrize("variant", ROW_VARIANTS, ids=[v[0] for v in ROW_VARIANTS])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,hidden", SHAPES)
def test_softmax_every_variant(cuda_device, variant, dtype, rows, hidden):
    dt = synth.dtype_of(dtype)
    plan = _row_plan(variant, "softmax", dt, hidden)
    if plan is None:
        pytest.skip("variant does not fit this width")
    x = synth.cast(synth.normal_np((rows, hidden), 871, std=3.0), dt)
    xd = x.to(cuda_device)
    yd = torch.empty_like(xd)
    A.check(A.ks_softmax_planned(yd.data_ptr(), xd.data_ptr(), rows, hidden, CODES[dt], plan,
                                 torch.cuda.current_stream().cuda_stream))
    ref, _ = oracle.softmax(x)
    compare_output(yd.cpu(), ref, dt, hidden, f"softmax {variant[0]} {dtype} [{rows},{hidden}]")


def _ln_check(out, ref, dt, h, name):
    away = ref.double().abs() > 0.05
    if dt != torch.float32 and bool(away.any()):
        assert int(ulp_dist(out[away], ref[away]).max()) <= 1, name
    rtol, atol = tol_for(dt, h)
    if dt == torch.float32:
        atol = rtol * 4.0
    ok, worst, _ = within_tol(out, ref, rtol, atol)
    assert ok, f"{name}: {worst}"


@pytest.mark.parametrize("variant", ROW_VARIANTS, ids=[v[0] for v in ROW_VARIANTS])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,hidden", SHAPES)
@pytest.mark.parametrize("affine", ["both", "none", "weight", "bias"])
def test_layer_norm_every_variant(cuda_device, variant, dtype, rows, hidden, affine):
    dt = synth.dtype_of(dtype)
    plan = _row_plan(variant, "layer_norm", dt, hidden)
    if plan is None:
        pytest.skip("variant does not fit this width")
    if affine in ("weight", "bias") and not plan.flags & A.KS_PLAN_AFFINE_SMEM:
        # one of the two rows: for the ring that holds them in shared memory, where the bias row
        # sits after the weight row only when there is one
        pytest.skip("weight-only and bias-only: the shared-memory affine ring")
    x = synth.cast(synth.normal_np((rows, hidden), 872) + 0.25, dt)
    w = synth.weight(hidden, dt) if affine in ("both", "weight") else None
    b = synth.cast(synth.normal_np((hidden,), 873, std=0.1), dt) if affine in ("both", "bias") else None
    xd = x.to(cuda_device)
    yd = torch.empty_like(xd)
    wd = w.to(cuda_device) if w is not None else None
    bd = b.to(cuda_device) if b is not None else None
    A.check(A.ks_layer_norm_planned(yd.data_ptr(), xd.data_ptr(),
                                    wd.data_ptr() if wd is not None else None,
                                    bd.data_ptr() if bd is not None else None, rows, hidden,
                                    1e-5, CODES[dt], plan, torch.cuda.current_stream().cuda_stream))
    ref, _ = oracle.layer_norm(x, w, b, 1e-5)
    _ln_check(yd.cpu(), ref, dt, hidden, f"layer_norm {variant[0]} {dtype} [{rows},{hidden}] {affine}")
    st, flags = A.ks_device_faults(clear=False)
    assert st == A.KS_SUCCESS and flags == 0


SILU_VARIANTS = [("flat256", A.KS_KERNEL_FLAT, 256), ("flat64", A.KS_KERNEL_FLAT, 64),
                 ("rows96", A.KS_KERNEL_CTA_ROW, 96), ("rows256", A.KS_KERNEL_CTA_ROW, 256),
                 ("rows32", A.KS_KERNEL_CTA_ROW, 32), ("scalar", A.KS_KERNEL_SCALAR, 256),
                 ("scalar96", A.KS_KERNEL_SCALAR, 96)]


@pytest.mark.parametrize("variant", SILU_VARIANTS, ids=[v[0] for v in SILU_VARIANTS])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,d", [(333, 512), (1001, 1000), (77, 3584), (5, 8192), (700, 64)])
def test_silu_and_mul_every_variant(cuda_device, variant, dtype, rows, d):
    dt = synth.dtype_of(dtype)
    name, kernel, block = variant
    if kernel != A.KS_KERNEL_SCALAR and (d * (4 if dt == torch.float32 else 2)) % 16:
        pytest.skip("vector kernel on a width that is not a whole number of vectors")
    plan = A.make_plan(kernel, 2, block)
    x = synth.cast(synth.normal_np((rows, 2 * d), 874, std=2.0), dt)
    xd = x.to(cuda_device)
    yd = torch.empty((rows, d), dtype=dt, device=cuda_device)
    A.check(A.ks_silu_and_mul_planned(yd.data_ptr(), xd.data_ptr(), rows, d, CODES[dt], plan,
                                      torch.cuda.current_stream().cuda_stream))
    ref, _ = oracle.silu_and_mul(x)
    compare_output(yd.cpu(), ref, dt, 8, f"silu_and_mul {name} {dtype} [{rows},{d}]")


def test_planned_equals_default_for_the_default_plan(cuda_device):
    """The plan ks_plan_launch reports, passed back through the planned entry point, gives the
    default entry point's bits."""
    import row_wise_rmsnorm_ks_gb300 as ks
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    s = torch.cuda.current_stream().cuda_stream
    for rows, hidden in [(1000, 576), (300, 8192), (40, 40000), (10, 1001)]:
        x = synth.cast(synth.normal_np((rows, hidden), 875, std=3.0), torch.bfloat16).to(cuda_device)
        st, p = A.ks_plan_launch(A.OP_SOFTMAX, rows, hidden, A.KS_DTYPE_BF16, True, sms, 0)
        assert st == A.KS_SUCCESS
        y = torch.empty_like(x)
        A.check(A.ks_softmax_planned(y.data_ptr(), x.data_ptr(), rows, hidden, A.KS_DTYPE_BF16, p, s))
        assert torch.equal(y, ks.softmax(x))
        st, p = A.ks_plan_launch(A.OP_LAYER_NORM, rows, hidden, A.KS_DTYPE_BF16, True, sms, 0)
        A.check(A.ks_layer_norm_planned(y.data_ptr(), x.data_ptr(), None, None, rows, hidden, 1e-5,
                                        A.KS_DTYPE_BF16, p, s))
        assert torch.equal(y, ks.layer_norm(x, None, None, 1e-5))
