"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by element, on the
same seeded inputs. Residual outputs must be bit-exact; normalised outputs within 1 ulp and the
stated tolerance (bf16 1e-2*|ref| + 1e-3, fp16 2e-3*|ref| + 1e-4).

Workloads follow the pages' shapes (Kernscope "CUDA performance", Triton Kernel Lab "Measured
Result" and "Decode Kernel Results", Triton Kernels "Benchmark results") widened to GB300 sizes;
the multi-gigabyte cases are compared on sampled rows plus properties checked on every row.
"""
import pytest
import torch

import oracle
import row_wise_rmsnorm_ks_gb300 as ks
from gpu_common import compare_output, record, run_and_check, sample_rows
from helpers import bits_equal, ulp_dist
from row_wise_rmsnorm_ks_gb300 import synth

pytestmark = pytest.mark.gpu


def test_small_bf16(cuda_device):
    run_and_check(synth.small(), cuda_device)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_medium_with_constant_and_zero_rows(cuda_device, dtype):
    w = synth.medium(dtype)
    out = run_and_check(w, cuda_device)
    y = out["y"].cpu()
    zi, ci, c = w.notes["zero_row"], w.notes["const_row"], w.notes["c"]
    assert (y[zi].double() == 0).all()
    # closed form for the constant row: c * w_j / sqrt(c^2 + eps), within 1 ulp
    eps32 = float(torch.tensor(w.eps, dtype=torch.float32))
    exact = (c * w.weight.double() / (c * c + eps32) ** 0.5)
    ref = oracle.encode(exact, w.dtype)
    assert int(ulp_dist(y[ci], ref).max()) <= 1


def test_fused_bf16(cuda_device):
    run_and_check(synth.fused(), cuda_device)


def test_fused_decode_shape(cuda_device):
    run_and_check(synth.decode(), cuda_device)


@pytest.mark.parametrize("rows", [1024, 4096, 32768])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
def test_prefill_sampled(cuda_device, op, rows):
    """The large prefill shape [rows, 8192] bf16, eps 1e-5 (rows up to 32768: 512 MiB a tensor),
    in the launch configuration the bench times. Sampled rows against the oracle; every row's
    residual against the rounded sum, computed independently with torch on the device."""
    w = synth.prefill_device(op, rows, 8192, "bf16", cuda_device)
    idx = sample_rows(rows)
    x_in = w.x.clone()
    r_in = w.residual.clone() if w.residual is not None else None
    out = run_and_check(w, cuda_device, rows_idx=idx, name=f"prefill {op} [{rows},8192]")
    if op != "rms_norm":
        assert bits_equal(out["r"], (x_in.float() + r_in.float()).to(torch.bfloat16))
    else:
        assert bool(torch.isfinite(out["y"].float()).all())


WIDE_H = [1536, 5120, 7168, 14336, 16384]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
@pytest.mark.parametrize("hidden", WIDE_H)
@pytest.mark.parametrize("rows", [1, 7, 333])
def test_wide_sweep_full(cuda_device, rows, hidden, op, dtype):
    """Heavy-tailed Student-t(3) rows, 1% of rows scaled by 1e3; every row compared."""
    w = synth.wide_device(op, hidden, rows, dtype, cuda_device)
    run_and_check(w, cuda_device, name=f"wide {op} {dtype} [{rows},{hidden}]")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
@pytest.mark.parametrize("hidden", WIDE_H)
def test_wide_sweep_65536_rows_sampled(cuda_device, hidden, op, dtype):
    rows = 65536
    w = synth.wide_device(op, hidden, rows, dtype, cuda_device)
    outl = w.notes["outlier_rows"]
    idx = sample_rows(rows, extra=outl[:16] + outl[-4:])
    x_in = w.x.clone()
    r_in = w.residual.clone() if w.residual is not None else None
    out = run_and_check(w, cuda_device, rows_idx=idx, name=f"wide {op} {dtype} [65536,{hidden}]")
    if op != "rms_norm":
        assert bits_equal(out["r"], (x_in.float() + r_in.float()).to(w.dtype))
    del x_in, r_in, out, w
    torch.cuda.empty_cache()


# ------------------------------------------------------------------------------ edge cases

EDGE_H = [1, 2, 3, 5, 7, 8, 16, 17, 64, 255, 1000, 1001, 4095, 4097, 12289, 20000, 40000]


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
@pytest.mark.parametrize("hidden", EDGE_H)
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
def test_edge_widths(cuda_device, hidden, dtype, op):
    """Ragged and odd widths (scalar path), widths around vector and team boundaries, and rows
    wider than the register-resident kernels hold."""
    rows = 5 if hidden < 20000 else 2
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, hidden), 31), dt)
    wt = synth.weight(hidden, dt)
    r = synth.cast(synth.normal_np((rows, hidden), 32), dt) if op != "rms_norm" else None
    w = synth.Workload(f"edge {op} {dtype} [{rows},{hidden}]", op, dt, x, wt, 1e-6, residual=r)
    run_and_check(w, cuda_device)


def _band_edges():
    """(dtype, op, hv) at every width where the launch heuristic's band table for many rows
    switches launch (a band's last width and the next one), from the committed measured record
    the table is generated from, plus both ends of the table."""
    import json
    import os

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "row_wise_rmsnorm_ks_gb300", "csrc", "bands",
                           "rms_norm_plan_bands.json")) as f:
        bands = bench.derive_plan_bands(json.load(f))
    out = []
    for key, bl in sorted(bands.items()):
        dt, op = key.split("/")
        hvs = {bench.PLAN_BAND_LO, bench.PLAN_BAND_HI}
        for hi, _, _ in bl[:-1]:
            hvs |= {hi, hi + 1}
        out += [(dt, op, hv) for hv in sorted(hvs)]
    return out


@pytest.mark.parametrize("dtype,op,hv", _band_edges())
@pytest.mark.parametrize("rows", [333, 701])
def test_default_plans_at_heuristic_edges(cuda_device, hv, op, dtype, rows):
    """The default entry points on many rows at every width where the launch heuristic switches
    plan, so each plan it can pick is checked: 333 rows (more than SMs, fewer than 4 per SM, so
    bands of the staged ring and the two-pass kernel take their one-pass fallback) and 701 (at
    least 4 per SM: those bands' own launch); both ragged."""
    dt = synth.dtype_of(dtype)
    hidden = hv * (4 if dt == torch.float32 else 8)
    x = synth.cast(synth.normal_np((rows, hidden), 41), dt)
    wt = synth.weight(hidden, dt)
    r = synth.cast(synth.normal_np((rows, hidden), 42, std=2.0), dt) if op != "rms_norm" else None
    w = synth.Workload(f"plan edge {op} {dtype} [{rows},{hidden}]", op, dt, x, wt, 1e-6,
                       residual=r)
    run_and_check(w, cuda_device)


def _wide_band_edges():
    """(dtype, op, hv) at every edge of the wide band table (rows of 2049..32768 vectors whose
    tensors exceed L2), from the committed measured record the table is generated from."""
    import json
    import os

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "row_wise_rmsnorm_ks_gb300", "csrc", "bands",
                           "rms_norm_wide_bands.json")) as f:
        bands = bench.derive_wide_bands(json.load(f))
    out = []
    for key, bl in sorted(bands.items()):
        dt, op = key.split("/")
        hvs = {bench.WIDE_LO, bench.WIDE_HI}
        for hi, _ in bl[:-1]:
            hvs |= {hi, hi + 1}
        out += [(dt, op, hv) for hv in sorted(hvs)]
    return out


@pytest.mark.parametrize("dtype,op,hv", _wide_band_edges())
def test_wide_band_edges(cuda_device, dtype, op, hv):
    """The default entry points at every width where the wide band table switches launch, with
    enough rows (ragged) that the tensors exceed L2, as the table requires: the staged kernel,
    the split and one-CTA two-pass kernels and the cluster kernel, each at its band's edges.
    Sampled rows against the oracle; the fused op's residual on every row against the rounded
    sum, computed with torch on the device."""
    dt = synth.dtype_of(dtype)
    hidden = hv * (4 if dt == torch.float32 else 8)
    rows = max(4 * 152 + 1, -(-(160 << 20) // (hv * 32)) + 3)
    w = synth.prefill_device(op, rows, hidden, dtype, cuda_device)
    x_in = w.x.clone()
    r_in = w.residual.clone() if w.residual is not None else None
    out = run_and_check(w, cuda_device, rows_idx=sample_rows(rows, k=12),
                        name=f"wide band edge {op} {dtype} [{rows},{hidden}]")
    if op != "rms_norm":
        assert bits_equal(out["r"], (x_in.float() + r_in.float()).to(dt))
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    st, flags = A.ks_device_faults(clear=True)
    assert st == A.KS_SUCCESS and flags == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
def test_unaligned_pointers(cuda_device, dtype, op):
    """Views starting one element into their storage are not 16-byte aligned: the scalar kernel
    must take them and give the same answers."""
    dt = synth.dtype_of(dtype)
    rows, hidden = 9, 1024
    base = synth.cast(synth.normal_np((rows * hidden + 1,), 41), dt).to(cuda_device)
    x = base[1:].view(rows, hidden)
    wbase = synth.weight(hidden + 1, dt).to(cuda_device)
    wt = wbase[1:]
    assert x.data_ptr() % 16 != 0 and wt.data_ptr() % 16 != 0
    x_host, w_host = x.cpu(), wt.cpu()
    if op == "rms_norm":
        y = ks.rms_norm(x, wt, 1e-6)
        ref, _ = oracle.rms_norm(x_host, w_host, 1e-6)
        compare_output(y.cpu(), ref, dt, hidden, f"unaligned {op} {dtype}")
    else:
        rbase = synth.cast(synth.normal_np((rows * hidden + 1,), 42), dt).to(cuda_device)
        r = rbase[1:].view(rows, hidden)
        r_host = r.cpu()
        ks.fused_add_rms_norm(x, r, wt, 1e-6)
        ref_x, ref_r, _ = oracle.fused_add_rms_norm(x_host, r_host, w_host, 1e-6)
        assert bits_equal(r.cpu(), ref_r)
        compare_output(x.cpu(), ref_x, dt, hidden, f"unaligned {op} {dtype}")


@pytest.mark.parametrize("hidden", [1024, 4096, 5000])
def test_in_place_plain(cuda_device, hidden):
    """out == x is allowed: each row is read completely before it is written."""
    x = synth.cast(synth.normal_np((64, hidden), 51), torch.bfloat16)
    wt = synth.weight(hidden, torch.bfloat16)
    ref, _ = oracle.rms_norm(x, wt, 1e-6)
    xd = x.to(cuda_device)
    y = ks.rms_norm(xd, wt.to(cuda_device), 1e-6, out=xd)
    assert y.data_ptr() == xd.data_ptr()
    compare_output(xd.cpu(), ref, torch.bfloat16, hidden, f"in-place rms_norm [64,{hidden}]")


def test_empty_and_batched_shapes(cuda_device):
    wt = synth.weight(64, torch.bfloat16).to(cuda_device)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda_device)
    assert ks.rms_norm(x, wt).shape == (0, 64)
    r = torch.empty_like(x)
    assert ks.fused_add_rms_norm(x, r, wt) is None
    # leading dimensions are flattened: Kernscope's (2, 3, 5)-style shapes
    x3 = synth.cast(synth.normal_np((2, 3, 64), 3), torch.bfloat16)
    y3 = ks.rms_norm(x3.to(cuda_device), wt).cpu()
    ref, _ = oracle.rms_norm(x3, wt.cpu())
    compare_output(y3, ref, torch.bfloat16, 64, "batched (2,3,64)")


def test_fused_with_zero_residual_equals_plain_on_gpu(cuda_device):
    """s = x + 0 = x, so the fused op computes the plain op's FP32 values: bit-identical results
    under one launch shape (one reduction order), and within 1 ulp under the two ops' default
    shapes, which the heuristic may pick differently."""
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    rows, hidden = 333, 4096
    x = synth.cast(synth.normal_np((rows, hidden), 61), torch.bfloat16).to(cuda_device)
    wt = synth.weight(hidden, torch.bfloat16).to(cuda_device)
    stream = torch.cuda.current_stream(cuda_device).cuda_stream
    for kernel, v, block, flags in ((A.KS_KERNEL_CTA_ROW, 4, 128, A.KS_PLAN_NO_PREFETCH),
                                    (A.KS_KERNEL_CTA_ROW, 2, 256, 0)):
        plan = A.make_plan(kernel, v, block, flags=flags)
        y = torch.empty_like(x)
        A.check(A.ks_rms_norm_planned(y.data_ptr(), x.data_ptr(), wt.data_ptr(), rows, hidden,
                                      1e-6, A.KS_DTYPE_BF16, plan, stream))
        xf, r = x.clone(), torch.zeros_like(x)
        A.check(A.ks_fused_add_rms_norm_planned(xf.data_ptr(), r.data_ptr(), wt.data_ptr(), rows,
                                                hidden, 1e-6, A.KS_DTYPE_BF16, plan, stream))
        assert bits_equal(xf.cpu(), y.cpu()) and bits_equal(r.cpu(), x.cpu())
    y = ks.rms_norm(x, wt)
    xf, r = x.clone(), torch.zeros_like(x)
    ks.fused_add_rms_norm(xf, r, wt)
    assert bits_equal(r.cpu(), x.cpu())
    assert int(ulp_dist(xf.cpu(), y.cpu()).max()) <= 1


def test_nonfinite_matches_oracle(cuda_device):
    x = torch.tensor([[1.0, float("inf"), 2.0, 3.0, 0.5, 0.25, 1.5, 2.5],
                      [1.0, float("nan"), 1.0, 1.0, 1.0, 1.0, 1.0, 1.0],
                      [1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0]], dtype=torch.float32)
    wt = torch.ones(8)
    y = ks.rms_norm(x.to(cuda_device), wt.to(cuda_device)).cpu()
    ref, _ = oracle.rms_norm(x, wt)
    assert bits_equal(y[:2], ref[:2])


def test_deterministic_and_guard_bands(cuda_device):
    """Two launches give identical bits; bytes just past the output are never written."""
    rows, hidden = 1000, 4096
    x = synth.cast(synth.normal_np((rows, hidden), 71), torch.bfloat16).to(cuda_device)
    wt = synth.weight(hidden, torch.bfloat16).to(cuda_device)
    buf = torch.full((rows * hidden + 4096,), 7.0, dtype=torch.bfloat16, device=cuda_device)
    out = buf[:rows * hidden].view(rows, hidden)
    ks.rms_norm(x, wt, out=out)
    y2 = ks.rms_norm(x, wt)
    assert bits_equal(out.cpu(), y2.cpu())
    assert (buf[rows * hidden:].float() == 7.0).all()
    record("guard bands", ok=True)


def test_rejects_requires_grad_and_cpu(cuda_device):
    x = torch.randn(4, 64, device=cuda_device, requires_grad=True)
    with pytest.raises(RuntimeError):
        ks.rms_norm(x, torch.ones(64, device=cuda_device))
    with pytest.raises(ValueError):
        ks.rms_norm(torch.randn(4, 64), torch.ones(64))


def test_overlap_rejected_before_launch(cuda_device):
    x = torch.randn(8, 64, device=cuda_device)
    with pytest.raises(ks.KsError) as e:
        ks.fused_add_rms_norm(x, x, torch.ones(64, device=cuda_device))
    assert e.value.name == "KS_ERR_OVERLAP"


def test_streams_are_honoured(cuda_device):
    """The launch goes to torch's current stream."""
    s = torch.cuda.Stream()
    x = synth.cast(synth.normal_np((256, 4096), 81), torch.bfloat16).to(cuda_device)
    wt = synth.weight(4096, torch.bfloat16).to(cuda_device)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        y = ks.rms_norm(x, wt)
    s.synchronize()
    ref, _ = oracle.rms_norm(x.cpu(), wt.cpu())
    compare_output(y.cpu(), ref, torch.bfloat16, 4096, "side stream")


# ------------------------------------------------- every kernel variant, via explicit plans

def _variant_plan(name, hidden, elem):
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    hv = hidden * elem // 16
    up32 = lambda n: -(-n // 32) * 32
    if name == "scalar":
        return A.make_plan(A.KS_KERNEL_SCALAR, 0, 256)
    if hidden * elem % 16:
        return None
    if name.startswith("twopass"):  # twopass_b<block>_u<vectors per step>
        block, u = name.split("_b")[1].split("_u")
        return A.make_plan(A.KS_KERNEL_TWOPASS_ROW, int(u), int(block))
    if name.startswith("split"):  # split[p]_c<cluster>_b<block>_u<vectors per step>
        c = int(name.split("_c")[1].split("_")[0])
        block, u = name.split("_b")[1].split("_u")
        if (c - 1) * -(-hv // c) >= hv:
            return None
        stages = 2 if name.startswith("splitp") else 0  # splitp: two rows in flight per cluster
        return A.make_plan(A.KS_KERNEL_TWOPASS_ROW, int(u), int(block), stages, cluster=c)
    flags = A.KS_PLAN_NO_PREFETCH if name.endswith("_np") else 0
    if name.startswith("warp_row"):
        v = next((v for v in (1, 2, 4, 6, 8) if 32 * v >= hv), None)
        return A.make_plan(A.KS_KERNEL_WARP_ROW, v, 128, flags=flags) if v else None
    v = 2 if name.startswith("cta_row_v2") else 4
    block = max(32, up32(-(-hv // v)))
    if block > (1024 if v == 2 else 512):
        return None
    if name.startswith("bulk_row"):  # bulk_row[_c<cluster>]_s<stages>[_v8][_m]
        stages = int(name.split("_s")[1].split("_")[0])
        if "_c" in name:  # the ring split over a cluster: each CTA stages its slice
            c = int(name.split("_c")[1].split("_")[0])
            vv = 8 if "_v8" in name else 4
            block = max(32, up32(-(-(-(-hv // c)) // vv)))
            if block > 512:
                return None
            # _m: the rows stay in shared memory, two in flight
            return A.make_plan(A.KS_KERNEL_BULK_ROW, vv, block, stages, cluster=c,
                               flags=A.KS_PLAN_SMEM_ROWS if name.endswith("_m") else 0)
        return A.make_plan(A.KS_KERNEL_BULK_ROW, 4, block, stages)
    if name.startswith("cluster_row"):
        c = int(name.split("_c")[1])
        block = max(32, up32(-(-(-(-hv // c)) // 4)))
        return A.make_plan(A.KS_KERNEL_CLUSTER_ROW, 4, block, cluster=c)
    return A.make_plan(A.KS_KERNEL_CTA_ROW, v, block, flags=flags)


VARIANTS = ["warp_row", "warp_row_np", "cta_row_v2", "cta_row_v2_np", "cta_row_v4",
            "cta_row_v4_np", "bulk_row_s1", "bulk_row_s2", "bulk_row_s5", "bulk_row_c2_s2",
            "bulk_row_c3_s1", "bulk_row_c8_s3", "bulk_row_c2_s2_v8", "bulk_row_c3_s3_v8",
            "bulk_row_c8_s4_v8", "bulk_row_c2_s2_m", "bulk_row_c3_s3_m", "bulk_row_c8_s4_m",
            "bulk_row_c2_s3_v8_m", "bulk_row_c4_s2_v8_m", "bulk_row_c8_s6_v8_m",
            "bulk_row_c16_s3_m", "bulk_row_c16_s2_v8_m",
            "cluster_row_c2", "cluster_row_c3",
            "cluster_row_c8", "twopass_b256_u4", "twopass_b512_u2", "twopass_b1024_u4",
            "twopass_b96_u2", "split_c2_b256_u4", "split_c3_b96_u2", "split_c4_b512_u2",
            "split_c8_b1024_u2", "splitp_c2_b256_u4", "splitp_c3_b96_u2", "splitp_c4_b512_u2",
            "splitp_c8_b1024_u2", "scalar"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
@pytest.mark.parametrize("rows,hidden", [(333, 1024), (1000, 1536), (77, 1400), (457, 4096),
                                         (300, 8192), (155, 16384)])
def test_every_kernel_variant_matches_oracle(cuda_device, variant, dtype, op, rows, hidden):
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    dt = synth.dtype_of(dtype)
    elem = 4 if dt == torch.float32 else 2
    plan = _variant_plan(variant, hidden, elem)
    if plan is None:
        pytest.skip("variant does not fit this width")
    if ("_v8" in variant or variant.endswith("_m")) and op != "rms_norm":
        pytest.skip("8 vectors per thread, rows kept in shared memory: the plain op's staged "
                    "kernel only")
    if plan.kernel == A.KS_KERNEL_BULK_ROW:
        hv = hidden * elem // 16
        stage = -(-hv // max(plan.cluster, 1)) * 16 * (2 if op != "rms_norm" else 1)
        if 128 + plan.stages * stage > 226 * 1024:
            pytest.skip("ring does not fit")
    x = synth.cast(synth.normal_np((rows, hidden), 91), dt)
    wt = synth.weight(hidden, dt)
    code = {torch.bfloat16: A.KS_DTYPE_BF16, torch.float16: A.KS_DTYPE_F16,
            torch.float32: A.KS_DTYPE_F32}[dt]
    xd, wd = x.to(cuda_device), wt.to(cuda_device)
    s = torch.cuda.current_stream().cuda_stream
    name = f"variant {variant} {op} {dtype} [{rows},{hidden}]"
    if op == "rms_norm":
        yd = torch.empty_like(xd)
        st = A.ks_rms_norm_planned(yd.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows, hidden,
                                   1e-6, code, plan, s)
        if st == A.KS_ERR_CUDA and plan.cluster > 8 and "resident" in A.ks_last_error():
            pytest.skip(f"the device places no cluster of {plan.cluster}")  # a non-portable size
        A.check(st)
        ref, _ = oracle.rms_norm(x, wt, 1e-6)
        compare_output(yd.cpu(), ref, dt, hidden, name)
    else:
        r = synth.cast(synth.normal_np((rows, hidden), 92, std=2.0), dt)
        rd = r.to(cuda_device)
        A.check(A.ks_fused_add_rms_norm_planned(xd.data_ptr(), rd.data_ptr(), wd.data_ptr(), rows,
                                                hidden, 1e-6, code, plan, s))
        ref_x, ref_r, _ = oracle.fused_add_rms_norm(x, r, wt, 1e-6)
        assert bits_equal(rd.cpu(), ref_r), name
        compare_output(xd.cpu(), ref_x, dt, hidden, name)
    st, flags = A.ks_device_faults(clear=True)
    assert st == A.KS_SUCCESS and flags == 0


@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
@pytest.mark.parametrize("dtype,hidden,rows", [("bf16", 20480, 200), ("bf16", 32768, 157),
                                               ("fp16", 24576, 100), ("fp32", 12288, 300),
                                               ("fp32", 16384, 77), ("bf16", 65536, 40),
                                               ("bf16", 131072, 21), ("bf16", 32768, 3),
                                               ("fp32", 20480, 5)])
def test_rows_wider_than_registers_match_oracle(cuda_device, op, dtype, hidden, rows):
    """Rows of more than 2048 vectors through the default heuristic: the two-pass kernel (split
    over a cluster for rows of more than 8192 vectors) with many rows, the register-resident
    cluster kernel with few."""
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    dt = synth.dtype_of(dtype)
    code = {torch.bfloat16: A.KS_DTYPE_BF16, torch.float16: A.KS_DTYPE_F16,
            torch.float32: A.KS_DTYPE_F32}[dt]
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    p = A.ks_plan_launch(0 if op == "rms_norm" else 1, rows, hidden, code, True, sms, 1)[1]
    assert p.kernel == A.KS_KERNEL_TWOPASS_ROW or (p.kernel == A.KS_KERNEL_CLUSTER_ROW
                                                    and p.cluster == 8)
    x = synth.cast(synth.student_t3_np((rows, hidden), 95), dt)
    wt = synth.weight(hidden, dt)
    xd, wd = x.to(cuda_device), wt.to(cuda_device)
    name = f"wide {op} {dtype} [{rows},{hidden}] {p.as_dict()['kernel_name']} c{p.cluster}"
    if op == "rms_norm":
        yd = ks.rms_norm(xd, wd, 1e-6)
        ref, _ = oracle.rms_norm(x, wt, 1e-6)
        compare_output(yd.cpu(), ref, dt, hidden, name)
    else:
        r = synth.cast(synth.normal_np((rows, hidden), 96, std=2.0), dt)
        rd = r.to(cuda_device)
        ks.fused_add_rms_norm(xd, rd, wd, 1e-6)
        ref_x, ref_r, _ = oracle.fused_add_rms_norm(x, r, wt, 1e-6)
        assert bits_equal(rd.cpu(), ref_r), name
        compare_output(xd.cpu(), ref_x, dt, hidden, name)
    st, flags = A.ks_device_faults(clear=True)
    assert st == A.KS_SUCCESS and flags == 0


@pytest.mark.parametrize("op,dtype,rows,hidden", [
    ("fused_add_rms_norm", "bf16", 1203, 65536),   # 8192 vectors: the split kernel, two rows in flight
    ("fused_add_rms_norm", "fp16", 605, 131072),   # 16384 vectors, cluster of 8
    ("rms_norm", "bf16", 701, 131072),             # 16384 vectors: the split kernel with L2 prefetch
    ("rms_norm", "fp32", 1001, 32768),             # 8192 fp32 vectors: one CTA per row
    ("fused_add_rms_norm", "fp32", 333, 65536)])   # 16384 fp32 vectors
def test_wide_rows_past_l2_through_the_heuristic(cuda_device, op, dtype, rows, hidden):
    """Many rows wider than 4096-8192 vectors whose tensors exceed L2, through the default entry
    points (the wide band table's staged or split kernels there), ragged row counts: sampled rows
    against the oracle, and the fused residual on every row against torch's rounded sum."""
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    dt = synth.dtype_of(dtype)
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    code = {torch.bfloat16: A.KS_DTYPE_BF16, torch.float16: A.KS_DTYPE_F16,
            torch.float32: A.KS_DTYPE_F32}[dt]
    p = A.ks_plan_launch(0 if op == "rms_norm" else 1, rows, hidden, code, True, sms, 1)[1]
    assert p.kernel in (A.KS_KERNEL_TWOPASS_ROW, A.KS_KERNEL_BULK_ROW) and p.cluster in (0, 2, 4, 8)
    x = synth.cast(synth.student_t3_dev((rows, hidden), 97, cuda_device), dt)
    wt = synth.weight(hidden, dt).to(cuda_device)
    idx = sample_rows(rows, k=12)
    name = f"wide past L2 {op} {dtype} [{rows},{hidden}] cluster {p.cluster} stages {p.stages}"
    if op == "rms_norm":
        y = ks.rms_norm(x, wt, 1e-6)
        ref, _ = oracle.rms_norm(x[idx].cpu(), wt.cpu(), 1e-6)
        compare_output(y[idx].cpu(), ref, dt, hidden, name)
    else:
        r = synth.cast(synth.normal_dev((rows, hidden), 98, cuda_device, std=2.0), dt)
        x_in, r_in = x.clone(), r.clone()
        ks.fused_add_rms_norm(x, r, wt, 1e-6)
        assert bits_equal(r, (x_in.float() + r_in.float()).to(dt)), name
        ref_x, ref_r, _ = oracle.fused_add_rms_norm(x_in[idx].cpu(), r_in[idx].cpu(), wt.cpu(), 1e-6)
        assert bits_equal(r[idx].cpu(), ref_r), name
        compare_output(x[idx].cpu(), ref_x, dt, hidden, name)
    st, flags = A.ks_device_faults(clear=True)
    assert st == A.KS_SUCCESS and flags == 0


def test_no_device_faults_recorded(cuda_device):
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    torch.cuda.synchronize()
    st, flags = A.ks_device_faults(clear=False)
    assert st == A.KS_SUCCESS and flags == 0


@pytest.mark.parametrize("cluster", [2, 4, 8])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
@pytest.mark.parametrize("rows,hidden", [(1, 16384), (7, 14336), (3, 5120), (500, 4096)])
def test_cluster_rows_wide_sweep(cuda_device, cluster, op, rows, hidden):
    """The cluster kernel on the wide sweep's heavy-tailed rows, few rows and many (grid capped
    to resident clusters, clusters striding over rows)."""
    from row_wise_rmsnorm_ks_gb300 import _abi as A
    w = synth.wide_device(op, hidden, rows, "bf16", cuda_device)
    hv = hidden // 8
    slice_vectors = -(-hv // cluster)
    threads = -(-slice_vectors // 4)
    block = max(32, -(-threads // 32) * 32)
    plan = A.make_plan(A.KS_KERNEL_CLUSTER_ROW, 4, block, cluster=cluster)
    s = torch.cuda.current_stream().cuda_stream
    x_host = w.x.cpu()
    wd = w.weight.to(cuda_device)
    name = f"cluster c{cluster} {op} [{rows},{hidden}]"
    if op == "rms_norm":
        y = torch.empty_like(w.x)
        A.check(A.ks_rms_norm_planned(y.data_ptr(), w.x.data_ptr(), wd.data_ptr(), rows, hidden,
                                      w.eps, A.KS_DTYPE_BF16, plan, s))
        ref, _ = oracle.rms_norm(x_host, w.weight.cpu(), w.eps)
        compare_output(y.cpu(), ref, torch.bfloat16, hidden, name)
    else:
        r_host = w.residual.cpu()
        A.check(A.ks_fused_add_rms_norm_planned(w.x.data_ptr(), w.residual.data_ptr(),
                                                wd.data_ptr(), rows, hidden, w.eps,
                                                A.KS_DTYPE_BF16, plan, s))
        ref_x, ref_r, _ = oracle.fused_add_rms_norm(x_host, r_host, w.weight.cpu(), w.eps)
        assert bits_equal(w.residual.cpu(), ref_r)
        compare_output(w.x.cpu(), ref_x, torch.bfloat16, hidden, name)
