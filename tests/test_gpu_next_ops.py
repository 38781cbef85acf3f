"""GPU parity of SwiGLU, Softmax and LayerNorm (through the C ABI) against the oracle.

Shapes from the pages: SwiGLU 8 x 2*4096 (Kernscope "Quick start"), 512 x 8192 in / 512 x 4096
out and rows 1..512 x widths 1024..8192 (Kernscope "SwiGLU baseline"), 128 x 1024 .. 2048 x 4096
(Triton Kernel Lab "Measured Result"); Softmax 512 x 128 .. 512 x 1024 (Kernscope "Softmax
measurements"), widths 1..16384 and a 65536-column fp16 row, non-finite rows (Kernscope
"Correctness"); LayerNorm on the RMSNorm shapes. Outputs within 1 ulp and the tolerance gate
(LayerNorm: 1 ulp away from zero, the gate near it, where the bias cancels).
"""
import pytest
import torch

import oracle
import row_wise_rmsnorm_ks_gb300 as ks
from gpu_common import compare_output, record
from helpers import tol_for, ulp_dist, within_tol
from row_wise_rmsnorm_ks_gb300 import _abi, synth

pytestmark = pytest.mark.gpu
DT = ["bf16", "fp16", "fp32"]


# ----------------------------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("rows,d", [(8, 4096), (512, 4096), (1, 1024), (16, 8192), (128, 1024),
                                    (3, 7), (5, 1), (33, 1001), (0, 16), (2048, 4096),
                                    # narrow rows, many of them: the flat walk crosses rows
                                    # inside a warp and leaves a ragged tail
                                    (3000, 8), (1000, 64), (777, 520), (20000, 96),
                                    (4099, 1408)])
def test_silu_and_mul(cuda_device, dtype, rows, d):
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, 2 * d), 801, std=2.0), dt)
    y = ks.silu_and_mul(x.to(cuda_device))
    assert y.shape == (rows, d)
    if rows:
        ref, _ = oracle.silu_and_mul(x)
        # fp32 bound (8+4)*2^-24: expf within 2 ulp plus three roundings
        compare_output(y.cpu(), ref, dt, 8, f"silu_and_mul {dtype} [{rows},{d}]")


def test_silu_and_mul_extremes_and_views(cuda_device):
    g = torch.tensor([[0.0, 30.0, -30.0, 100.0, -100.0, float("inf"), float("-inf"), 2.0]])
    up = torch.tensor([[7.0, 3.0, 5.0, -2.0, 4.0, 1.0, 1.0, 0.0]])
    x = torch.cat([g, up], dim=1)
    y = ks.silu_and_mul(x.to(cuda_device)).cpu()
    ref, _ = oracle.silu_and_mul(x)
    assert torch.equal(torch.isnan(y), torch.isnan(ref))
    fin = ~torch.isnan(ref)
    ok, worst, _ = within_tol(y[fin], ref[fin], 1e-6, 1e-30)
    assert ok, worst
    # a contiguous view that starts one element in: unaligned, scalar path
    base = synth.cast(synth.normal_np((4 * 2 * 64 + 1,), 5), torch.bfloat16).to(cuda_device)
    xv = base[1:].view(4, 128)
    yv = ks.silu_and_mul(xv).cpu()
    refv, _ = oracle.silu_and_mul(xv.cpu())
    compare_output(yv, refv, torch.bfloat16, 1, "silu_and_mul unaligned view")


# ----------------------------------------------------------------------------------- Softmax

@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("rows,h", [(512, 1024), (512, 128), (2, 5), (7, 1), (3, 63), (100, 4096),
                                    (4, 16384), (33, 1000), (0, 8), (64, 2048)])
def test_softmax(cuda_device, dtype, rows, h):
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, h), 802, std=3.0), dt)
    y = ks.softmax(x.to(cuda_device))
    if rows:
        ref, _ = oracle.softmax(x)
        compare_output(y.cpu(), ref, dt, h, f"softmax {dtype} [{rows},{h}]")


def test_softmax_wide_fp16(cuda_device):
    x = synth.cast(synth.normal_np((3, 65536), 803), torch.float16)
    y = ks.softmax(x.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(x)
    compare_output(y, ref, torch.float16, 65536, "softmax fp16 [3,65536]")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("h", [8, 1000])
def test_softmax_nonfinite_rows(cuda_device, dtype, h):
    dt = synth.dtype_of(dtype)
    x = synth.normal_np((6, h), 804)
    inf, nan = float("inf"), float("nan")
    x[0, 1] = -inf; x[0, 3] = -inf        # masked entries
    x[1, 2] = nan                          # NaN row
    x[2, 0] = inf                          # +inf row
    x[3, :] = -inf                         # all -inf row
    x[4, :] = 0.0                          # uniform row
    xt = synth.cast(x, dt)
    y = ks.softmax(xt.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(xt)
    assert torch.equal(torch.isnan(y), torch.isnan(ref))
    assert torch.isnan(y[1:4]).all() and (y[0, [1, 3]] == 0).all()
    fin = ~torch.isnan(ref)
    rtol, atol = tol_for(dt, h)
    assert within_tol(y[fin], ref[fin], rtol, atol)[0]


def test_softmax_in_place(cuda_device):
    x = synth.cast(synth.normal_np((64, 4096), 805), torch.bfloat16)
    ref, _ = oracle.softmax(x)
    xd = x.to(cuda_device)
    ks.softmax(xd, out=xd)
    compare_output(xd.cpu(), ref, torch.bfloat16, 4096, "softmax in place")


# --------------------------------------------------------------------------------- LayerNorm

def _ln_check(out, ref, dt, h, name):
    away = ref.double().abs() > 0.05
    if dt != torch.float32 and bool(away.any()):
        assert int(ulp_dist(out[away], ref[away]).max()) <= 1, name
    rtol, atol = tol_for(dt, h)
    if dt == torch.float32:
        # fp32: the mean's rounding error (about H * 2^-24 * |mean|) moves every output by
        # itself times rstd, whatever the output's size: an absolute term of the same order
        atol = rtol * 4.0
    ok, worst, _ = within_tol(out, ref, rtol, atol)
    record(name, worst_excess=worst, n=out.numel())
    assert ok, f"{name}: {worst}"


AFFINE = ["both", "none", "weight", "bias"]  # each combination is its own kernel instantiation


def _affine(affine, h, dt, seed):
    w = synth.weight(h, dt) if affine in ("both", "weight") else None
    b = synth.cast(synth.normal_np((h,), seed, std=0.1), dt) if affine in ("both", "bias") else None
    return w, b


def _dev(t, device):
    return t.to(device) if t is not None else None


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("rows,h", [(128, 1024), (2048, 4096), (512, 4096), (4, 1536), (333, 8192),
                                    (7, 16384), (5, 17), (3, 1000), (2, 20000)])
@pytest.mark.parametrize("affine", AFFINE)
def test_layer_norm(cuda_device, dtype, rows, h, affine):
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, h), 806) + 0.25, dt)
    w, b = _affine(affine, h, dt, 807)
    y = ks.layer_norm(x.to(cuda_device), _dev(w, cuda_device), _dev(b, cuda_device), 1e-5).cpu()
    ref, _ = oracle.layer_norm(x, w, b, 1e-5)
    _ln_check(y, ref, dt, h, f"layer_norm {dtype} [{rows},{h}] affine={affine}")


def test_layer_norm_constant_row_and_in_place(cuda_device):
    h = 4096
    x = synth.cast(synth.normal_np((16, h), 808), torch.bfloat16)
    x[3] = 0.75
    w = synth.weight(h, torch.bfloat16)
    b = synth.cast(synth.normal_np((h,), 809), torch.bfloat16)
    ref, _ = oracle.layer_norm(x, w, b, 1e-5)
    xd = x.to(cuda_device)
    ks.layer_norm(xd, w.to(cuda_device), b.to(cuda_device), 1e-5, out=xd)
    y = xd.cpu()
    assert torch.equal(y[3].float(), b.float())       # constant row: exactly the bias
    _ln_check(y, ref, torch.bfloat16, h, "layer_norm in place")


def test_next_ops_reject_bad_arguments(cuda_device):
    x = torch.randn(4, 8, device=cuda_device)
    assert _abi.ks_silu_and_mul(x.data_ptr(), x.data_ptr(), 4, 4, _abi.KS_DTYPE_F32, None) == \
        _abi.KS_ERR_OVERLAP
    assert _abi.ks_softmax(x.data_ptr(), x.data_ptr(), 4, 0, _abi.KS_DTYPE_F32, None) == \
        _abi.KS_ERR_INVALID_ARGUMENT
    assert _abi.ks_layer_norm(x.data_ptr(), x.data_ptr(), None, None, 4, 8, 0.0,
                              _abi.KS_DTYPE_F32, None) == _abi.KS_ERR_INVALID_ARGUMENT
    with pytest.raises(ValueError):
        ks.silu_and_mul(torch.randn(4, 7, device=cuda_device))
    st, flags = _abi.ks_device_faults(clear=False)
    assert st == _abi.KS_SUCCESS and flags == 0


@pytest.mark.parametrize("dtype", DT)
def test_softmax_extreme_spread(cuda_device, dtype):
    """exp(z) down to fp32 subnormals (z to -103): bf16 keeps fp32's exponent range, so tiny
    probabilities survive the cast and must still be within the gate."""
    dt = synth.dtype_of(dtype)
    row = [0.0, -1.0, -20.0, -50.0, -87.0, -88.0, -90.0, -95.0, -100.0, -103.0, -3.0, -0.5,
           -60.0, -70.0, -80.0, -86.0]
    x = synth.cast(torch.tensor([row, [v / 2 for v in row]], dtype=torch.float32), dt)
    y = ks.softmax(x.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(x)
    compare_output(y, ref, dt, 16, f"softmax extreme spread {dtype}")


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("h", [1024, 4096, 8192, 10240, 12288, 16384])
@pytest.mark.parametrize("affine", AFFINE)
def test_layer_norm_many_rows_staged(cuda_device, dtype, h, affine):
    """Enough rows (>= 4 rows per SM) for the staged ring, or, for rows of 1024..2047 vectors,
    the wide kernel's 128-thread CTAs: every row against the oracle, and the ring's fault word
    stays clear."""
    dt = synth.dtype_of(dtype)
    rows = 1000
    x = synth.cast(synth.normal_np((rows, h), 811) - 0.5, dt)
    w, b = _affine(affine, h, dt, 812)
    y = ks.layer_norm(x.to(cuda_device), _dev(w, cuda_device), _dev(b, cuda_device), 1e-5).cpu()
    ref, _ = oracle.layer_norm(x, w, b, 1e-5)
    _ln_check(y, ref, dt, h, f"layer_norm staged {dtype} [{rows},{h}] affine={affine}")
    st, flags = _abi.ks_device_faults(clear=False)
    assert st == _abi.KS_SUCCESS and flags == 0


# --------------------------------------------------------------- rows wider than 2048 vectors

@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("rows,h", [(300, 20480), (97, 65536), (5, 40000)])
def test_softmax_rows_wider_than_registers(cuda_device, dtype, rows, h):
    """The wide multi-pass kernel (max, sum, outputs; later passes from L2)."""
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, h), 831, std=3.0), dt)
    y = ks.softmax(x.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(x)
    compare_output(y, ref, dt, h, f"softmax wide {dtype} [{rows},{h}]")


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("rows,h", [(300, 20480), (97, 65536), (5, 40000)])
@pytest.mark.parametrize("affine", AFFINE)
def test_layer_norm_rows_wider_than_registers(cuda_device, dtype, rows, h, affine):
    """The wide multi-pass kernel (mean, variance, outputs; later passes from L2)."""
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, h), 832) + 0.5, dt)
    w, b = _affine(affine, h, dt, 833)
    y = ks.layer_norm(x.to(cuda_device), _dev(w, cuda_device), _dev(b, cuda_device), 1e-5).cpu()
    ref, _ = oracle.layer_norm(x, w, b, 1e-5)
    _ln_check(y, ref, dt, h, f"layer_norm wide {dtype} [{rows},{h}] affine={affine}")
    st, flags = _abi.ks_device_faults(clear=False)
    assert st == _abi.KS_SUCCESS and flags == 0


# ------------------------------------------- plan bands: warp rows and the SwiGLU launch shapes

# Row widths in 16-byte vectors at the edges of the measured plan bands for many rows (warp rows
# at 2, 4, 6 or 8 vectors per lane, CTA rows, the general rule), for every dtype.
BAND_HV = [1, 2, 7, 8, 9, 12, 13, 16, 17, 20, 21, 28, 29, 32, 33, 40, 41, 44, 45, 52, 53, 54,
           56, 57, 63, 64, 65, 72, 73, 80, 81, 82, 96, 97, 112, 113, 127, 128, 129, 130, 144, 145,
           168, 169, 170, 176, 177, 178, 192, 193, 208, 209, 216, 217, 224, 225, 226, 256, 257]


def _elems(dt, hv):
    return hv * (4 if dt == torch.float32 else 8)


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("hv", BAND_HV)
def test_softmax_at_plan_band_edges(cuda_device, dtype, hv):
    """Many rows (1001: more than SMs, not a multiple of a CTA's 4 warp rows) at each band edge;
    also one row with NaN, +inf, all -inf and masked entries, which the warp kernels must treat
    as the CTA kernels do."""
    dt = synth.dtype_of(dtype)
    h = _elems(dt, hv)
    x = synth.normal_np((1001, h), 810, std=3.0)
    inf, nan = float("inf"), float("nan")
    x[5, 1] = -inf; x[5, 3] = -inf         # masked entries
    x[6, 2] = nan                            # NaN row
    x[7, 0] = inf                            # +inf row
    x[8, :] = -inf                           # all -inf row
    # torch's cast keeps the infinities (the input recipe's fp16 cast saturates them)
    xt = torch.tensor(x, dtype=torch.float32).to(dt)
    y = ks.softmax(xt.to(cuda_device)).cpu()
    ref, _ = oracle.softmax(xt)
    assert torch.equal(torch.isnan(y), torch.isnan(ref))
    assert torch.isnan(y[6:9]).all() and (y[5, [1, 3]] == 0).all()
    fin = ~torch.isnan(ref).any(dim=1)
    compare_output(y[fin], ref[fin], dt, h, f"softmax band {dtype} [1001,{h}]")


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("hv", BAND_HV)
@pytest.mark.parametrize("affine", AFFINE)
def test_layer_norm_at_plan_band_edges(cuda_device, dtype, hv, affine):
    dt = synth.dtype_of(dtype)
    h = _elems(dt, hv)
    x = synth.cast(synth.normal_np((1001, h), 811) + 0.25, dt)
    x[9] = 0.75  # a constant row
    w, b = _affine(affine, h, dt, 812)
    y = ks.layer_norm(x.to(cuda_device), _dev(w, cuda_device), _dev(b, cuda_device), 1e-5).cpu()
    ref, _ = oracle.layer_norm(x, w, b, 1e-5)
    _ln_check(y, ref, dt, h, f"layer_norm band {dtype} [1001,{h}] affine={affine}")


def _wide_band_edges():
    """(op, dtype, hv) at every edge of the Softmax and LayerNorm width bands past 256 vectors
    (each band's last width and the next), from the committed measured record the band tables
    are generated from."""
    import json
    import os

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "row_wise_rmsnorm_ks_gb300", "csrc", "bands",
                           "softmax_layer_norm_bands.json")) as f:
        rec = json.load(f)
    out = set()
    for _, op, dts in bench.OPS_BAND_TABLES:
        bands = bench.derive_bands(rec, op, dts)
        for hi, *_ in bands[:-1]:
            if hi >= 256:
                for dt in dts:
                    out |= {(op, dt, hi), (op, dt, hi + 1)}
    return sorted(out)


@pytest.mark.parametrize("op,dtype,hv", _wide_band_edges())
def test_wide_band_edges(cuda_device, op, dtype, hv):
    """Many rows (1001: at least 4 per SM, so the ring and wide-kernel bands apply) at each edge of
    the bands past 256 vectors; LayerNorm with weight and bias and a constant row."""
    dt = synth.dtype_of(dtype)
    h = _elems(dt, hv)
    if op == "softmax":
        x = synth.cast(synth.normal_np((1001, h), 814, std=3.0), dt)
        y = ks.softmax(x.to(cuda_device)).cpu()
        ref, _ = oracle.softmax(x)
        compare_output(y, ref, dt, h, f"softmax wide band edge {dtype} hv={hv}")
    else:
        x = synth.cast(synth.normal_np((1001, h), 815) + 0.25, dt)
        x[9] = 0.75  # a constant row
        w, b = _affine("both", h, dt, 816)
        y = ks.layer_norm(x.to(cuda_device), _dev(w, cuda_device), _dev(b, cuda_device), 1e-5).cpu()
        ref, _ = oracle.layer_norm(x, w, b, 1e-5)
        _ln_check(y, ref, dt, h, f"layer_norm wide band edge {dtype} hv={hv}")
    st, flags = _abi.ks_device_faults(clear=False)
    assert st == _abi.KS_SUCCESS and flags == 0


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("dv", [16, 31, 32, 33, 64, 96, 128, 159, 160, 161, 191, 192, 193, 256, 287,
                                288, 447, 448, 512, 576, 640, 1024, 1280, 2048])
def test_silu_and_mul_at_plan_band_edges(cuda_device, dtype, dv):
    """SwiGLU on many rows at the edges of its launch shapes: the flat walk, and the row kernel
    with its CTAs fitted to the row (at most 256 threads, the fewest idle)."""
    dt = synth.dtype_of(dtype)
    d = _elems(dt, dv)
    rows = 700 if dv <= 512 else 150
    x = synth.cast(synth.normal_np((rows, 2 * d), 813, std=2.0), dt)
    y = ks.silu_and_mul(x.to(cuda_device)).cpu()
    ref, _ = oracle.silu_and_mul(x)
    compare_output(y, ref, dt, 8, f"silu_and_mul band {dtype} [{rows},{d}]")
