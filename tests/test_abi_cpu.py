"""The C-ABI boundary on CPU (no GPU needed): libks builds for sm_103a, loads, exports every
symbol include/ks.h declares, and rejects invalid calls with the documented status before any
CUDA call. Only invalid calls are made here: a valid call would launch a kernel.

Also the host-side launch heuristic (after Triton Kernels' CPU tests of its launch-config
heuristics, "Running the tests"), checked through ks_plan_launch.
"""
import os
import re
import subprocess

import pytest

from row_wise_rmsnorm_ks_gb300 import _abi
from row_wise_rmsnorm_ks_gb300 import build as ks_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ks.h")

BF16, F16, F32 = _abi.KS_DTYPE_BF16, _abi.KS_DTYPE_F16, _abi.KS_DTYPE_F32
FAKE = 0x10000  # a non-NULL address that is never dereferenced (every call below fails first)


@pytest.fixture(scope="module", autouse=True)
def lib():
    ks_build.build()
    return _abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ks_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_exactly_the_binding_surface():
    assert declared_functions() == sorted(_abi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ks_build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ks_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_is_built_for_sm103a():
    with open(os.path.join(ks_build.OUT_DIR, "ptxas_report.txt")) as f:
        rep = f.read()
    assert "for 'sm_103a'" in rep
    assert "rows_vec_kernel" in rep and "rows_scalar_kernel" in rep


def test_status_strings():
    names = ["KS_SUCCESS", "KS_ERR_INVALID_ARGUMENT", "KS_ERR_UNSUPPORTED_DTYPE",
             "KS_ERR_OVERLAP", "KS_ERR_CUDA"]
    for code, name in enumerate(names):
        assert _abi.ks_status_string(code) == name
    assert _abi.ks_status_string(99) == "KS_UNKNOWN_STATUS"
    assert _abi.ks_version() >= 100


@pytest.mark.parametrize("fused", [False, True])
def test_invalid_arguments_rejected_before_any_cuda_call(fused):
    call = _abi.ks_fused_add_rms_norm if fused else _abi.ks_rms_norm
    a, b, w = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    assert call(a, b, w, 4, 0, 1e-6, BF16, None) == E            # hidden == 0
    assert call(a, b, w, 4, -3, 1e-6, BF16, None) == E           # hidden < 0
    assert call(a, b, w, -1, 64, 1e-6, BF16, None) == E          # rows < 0
    for eps in (0.0, -1e-6, float("nan"), float("inf")):
        assert call(a, b, w, 4, 64, eps, BF16, None) == E, eps   # eps not finite and > 0
    assert call(0, b, w, 4, 64, 1e-6, BF16, None) == E           # NULL with rows > 0
    assert call(a, 0, w, 4, 64, 1e-6, BF16, None) == E
    assert call(a, b, 0, 4, 64, 1e-6, BF16, None) == E
    assert call(a, b, w, 1 << 62, 1 << 20, 1e-6, BF16, None) == E  # byte size overflows
    assert "eps" in _abi.ks_last_error() or "overflow" in _abi.ks_last_error()
    assert call(a, b, w, 4, 64, 1e-6, 7, None) == _abi.KS_ERR_UNSUPPORTED_DTYPE
    assert call(a, b, w, 4, 64, 1e-6, -1, None) == _abi.KS_ERR_UNSUPPORTED_DTYPE


@pytest.mark.parametrize("fused", [False, True])
def test_empty_input_is_success_without_launch(fused):
    call = _abi.ks_fused_add_rms_norm if fused else _abi.ks_rms_norm
    # rows == 0: legal, nothing launched, pointers may be NULL
    assert call(0, 0, 0, 0, 64, 1e-6, BF16, None) == _abi.KS_SUCCESS


def test_overlap_rules_fused():
    rows, hidden, e = 4, 64, 2
    n = rows * hidden * e
    x, w = FAKE, FAKE + 10 * n
    O = _abi.KS_ERR_OVERLAP
    assert _abi.ks_fused_add_rms_norm(x, x, w, rows, hidden, 1e-6, BF16, None) == O
    assert _abi.ks_fused_add_rms_norm(x, x + n - 2, w, rows, hidden, 1e-6, BF16, None) == O
    assert _abi.ks_fused_add_rms_norm(x, x + 5 * n, x + 2, rows, hidden, 1e-6, BF16, None) == O
    assert _abi.ks_fused_add_rms_norm(x, x + 5 * n, x + 5 * n + 64, rows, hidden, 1e-6, BF16,
                                      None) == O
    assert "overlap" in _abi.ks_last_error()


def test_overlap_rules_plain():
    rows, hidden, e = 4, 64, 2
    n = rows * hidden * e
    x, w = FAKE, FAKE + 10 * n
    O = _abi.KS_ERR_OVERLAP
    assert _abi.ks_rms_norm(x + 2, x, w, rows, hidden, 1e-6, BF16, None) == O   # partial overlap
    assert _abi.ks_rms_norm(w - 2, x, w, rows, hidden, 1e-6, BF16, None) == O   # out over weight


# -------------------------------------------------------------------------- plan heuristic

def plan(op, rows, hidden, dtype=BF16, aligned=True, sms=152, bps=0):
    st, p = _abi.ks_plan_launch(op, rows, hidden, dtype, aligned, sms, bps)
    assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
    return p


@pytest.mark.parametrize("op,hidden,dtype,v", [(0, 256, BF16, 1), (0, 512, BF16, 2), (0, 768, F16, 4),
                                               (1, 768, BF16, 4), (0, 384, F32, 4)])
def test_few_narrow_rows_take_warp_per_row(op, hidden, dtype, v):
    p = plan(op, 100, hidden, dtype)  # at most SMs rows: a warp per row, one row per CTA
    assert p.kernel == _abi.KS_KERNEL_WARP_ROW and p.vec_per_thread == v and p.team == 32
    assert p.block == 32 and p.grid == 100


NO_PF = _abi.KS_PLAN_NO_PREFETCH
CTA, BULK, TWO = _abi.KS_KERNEL_CTA_ROW, _abi.KS_KERNEL_BULK_ROW, _abi.KS_KERNEL_TWOPASS_ROW
WARP = _abi.KS_KERNEL_WARP_ROW
# (Many rows of 97..2048 vectors take the measured band table: tests/test_plan_bands_cpu.py.)


def test_few_rows_keep_the_latency_rules():
    # rows <= SMs: the exceptions above apply only to many rows
    assert plan(0, 100, 1024, BF16).kernel == _abi.KS_KERNEL_WARP_ROW
    p = plan(0, 100, 4096, BF16)
    assert p.kernel == _abi.KS_KERNEL_CTA_ROW and p.vec_per_thread == 2


def test_warp_per_row_spreads_few_rows_over_sms():
    p = plan(0, 128, 1024)
    assert p.block == 32 and p.grid == 128  # 128 rows on 128 SMs


def test_latency_regime_keeps_one_row_per_cta_plans():
    p = plan(1, 100, 8192)  # fused, few rows: 4 vectors, prefetch on (nothing to fetch)
    assert p.kernel == CTA and p.vec_per_thread == 4 and p.flags == 0
    p = plan(0, 100, 8192)  # plain, <= 1024 vectors: 2 vectors per thread
    assert p.kernel == CTA and p.vec_per_thread == 2 and p.block == 512
    p = plan(1, 4, 16384)  # fused, widest rows, few rows: a cluster of 8 CTAs per row
    assert p.kernel == _abi.KS_KERNEL_CLUSTER_ROW and p.cluster == 8


def test_fp32_counts_four_elements_per_vector():
    # 4096 fp32 = 1024 vectors: few rows take 2 vectors per thread (512 threads)
    p = plan(0, 10, 4096, dtype=F32)
    assert p.kernel == _abi.KS_KERNEL_CTA_ROW and p.block == 512 and p.vec_per_thread == 2
    # many rows of 1024 fp32 = 256 vectors: whatever launch the band table names covers exactly
    # 256 vectors (a warp at 8 vectors per lane, or a CTA with no idle warp)
    for op in (0, 1):
        p = plan(op, 32768, 1024, dtype=F32)
        if p.kernel == _abi.KS_KERNEL_WARP_ROW:
            assert p.vec_per_thread == 8
        else:
            assert p.kernel == CTA and p.block * p.vec_per_thread == 256


@pytest.mark.parametrize("hidden,aligned", [(17, True), (1001, True), (4096, False),
                                            (20004, True), (140001, True)])
def test_scalar_fallback(hidden, aligned):
    p = plan(1, 7, hidden, aligned=aligned)
    assert p.kernel == _abi.KS_KERNEL_SCALAR
    assert p.block % 32 == 0 and 32 <= p.block <= 1024


def test_persistent_grid_is_capped_by_residency():
    p = plan(0, 32768, 8192, bps=2)
    assert p.grid == 304 and p.rows_per_pass == 304
    p = plan(0, 100, 8192, bps=2)
    assert p.grid == 100
    p = plan(0, 32768, 1024, F16, bps=3)  # warp per row: 8 rows per CTA
    assert p.grid == 152 * 3 and p.rows_per_pass == 152 * 3 * 8


def test_empty_plan_and_bad_arguments():
    assert plan(0, 0, 64).kernel == _abi.KS_KERNEL_NONE
    st, _ = _abi.ks_plan_launch(5, 1, 64, BF16, True, 152, 0)
    assert st == _abi.KS_ERR_INVALID_ARGUMENT
    st, _ = _abi.ks_plan_launch(0, 1, 0, BF16, True, 152, 0)
    assert st == _abi.KS_ERR_INVALID_ARGUMENT
    st, _ = _abi.ks_plan_launch(0, 1, 64, 5, True, 152, 0)
    assert st == _abi.KS_ERR_UNSUPPORTED_DTYPE


@pytest.mark.parametrize("dtype", [BF16, F16, F32])
def test_plan_invariants_over_a_sweep(dtype):
    e = 4 if dtype == F32 else 2
    for hidden in [1, 3, 8, 64, 100, 128, 1000, 1024, 1536, 2048, 3000, 4096, 8192, 12288,
                   16384, 16392, 32768, 100000]:
        for rows in [1, 7, 152, 333, 65536]:
            p = plan(1, rows, hidden, dtype=dtype, bps=2)
            assert p.block % 32 == 0 and 32 <= p.block <= 1024
            assert 1 <= p.grid <= max(rows, 1) * max(p.cluster, 1)
            if p.kernel == _abi.KS_KERNEL_TWOPASS_ROW:
                assert hidden * e % 16 == 0 and p.vec_per_thread in (2, 4)
            elif p.kernel in (_abi.KS_KERNEL_WARP_ROW, _abi.KS_KERNEL_CTA_ROW,
                              _abi.KS_KERNEL_BULK_ROW, _abi.KS_KERNEL_CLUSTER_ROW):
                assert hidden * e % 16 == 0
                assert p.team * p.vec_per_thread * (16 // e) >= hidden
                if p.kernel != _abi.KS_KERNEL_WARP_ROW:
                    assert p.block <= (1024 if p.vec_per_thread <= 2 else 512)
                if p.kernel == _abi.KS_KERNEL_CLUSTER_ROW:
                    assert p.grid % p.cluster == 0 and 2 <= p.cluster <= 8
                if p.kernel == _abi.KS_KERNEL_BULK_ROW:
                    assert p.smem_bytes <= 226 * 1024 and p.stages >= 2
                    assert p.cluster == 0 or (p.grid % p.cluster == 0 and 2 <= p.cluster <= 8)


@pytest.mark.parametrize("hidden,dtype", [(20000, BF16), (32768, BF16), (65536, BF16),
                                          (131072, BF16), (140000, BF16), (12288, F32),
                                          (16384, F32), (32768, F32)])
def test_wide_rows_outside_the_band_table(hidden, dtype):
    """Rows wider than 2048 vectors that the wide band table does not cover (it takes many rows,
    at least 4 per SM, whose tensors exceed L2; tests/test_plan_bands_cpu.py checks it): rows
    that fit in L2 take one CTA per row and two passes, with a grid that keeps the rows in flight
    within L2; three rows take the register-resident cluster kernel."""
    e = 4 if dtype == F32 else 2
    hv = hidden * e // 16
    for op in (0, 1):
        rows = max(153, (100 << 20) // (hv * 32))  # more rows than SMs, x and y within L2
        if rows * hv * 32 > (128 << 20):
            continue
        p = plan(op, rows, hidden, dtype=dtype, bps=1)
        assert p.kernel == _abi.KS_KERNEL_TWOPASS_ROW and p.cluster == 0
        assert p.vec_per_thread == (4 if (not op or (dtype == F32 and hv <= 2048)) else 2)
        assert p.team == p.block and p.flags == _abi.KS_PLAN_NO_PREFETCH
        # the grid keeps the rows in flight within 96 MiB of L2, but takes at least every SM
        assert p.grid == min(rows, 152, max(152, (96 << 20) // (hv * 16 * (2 if op else 1))))
        # few rows: the register-resident cluster kernel, 8 CTAs per row (up to 16384 vectors)
        p = plan(op, 3, hidden, dtype=dtype, bps=1)
        if hv <= 16384:
            assert p.kernel == _abi.KS_KERNEL_CLUSTER_ROW and p.cluster == 8
            assert p.block * p.vec_per_thread * 8 >= hv and p.grid == 24
        else:
            assert p.kernel == _abi.KS_KERNEL_TWOPASS_ROW and p.grid == 3


@pytest.mark.parametrize("op", [0, 1])
def test_rows_past_the_wide_table_take_the_split_kernel(op):
    """Many rows wider than 32768 vectors whose tensors exceed L2: the two-pass kernel split over
    a cluster of 8 CTAs (plain: slice prefetch, one row in flight; fused: two rows in flight),
    whole clusters, each with the same number of rows."""
    hidden, hv, rows = 300000, 37500, 4096
    p = plan(op, rows, hidden, dtype=BF16, bps=1)
    assert p.kernel == _abi.KS_KERNEL_TWOPASS_ROW and p.cluster == 8
    assert p.team == p.block * 8 and p.block == (512 if op else 256)
    assert p.flags == (_abi.KS_PLAN_NO_PREFETCH if op else 0) and p.stages == (2 if op else 0)
    n = min(152 // 8, (96 << 20) // (hv * 16 * (4 if op else 1)))
    waves = -(-rows // n)
    assert p.grid == -(-rows // waves) * 8


def test_two_pass_plans_are_checked():
    a, b, w = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    mk = _abi.make_plan
    for p in (mk(_abi.KS_KERNEL_TWOPASS_ROW, 3, 256), mk(_abi.KS_KERNEL_TWOPASS_ROW, 4, 2048),
              mk(_abi.KS_KERNEL_TWOPASS_ROW, 4, 100)):
        assert _abi.ks_rms_norm_planned(a, b, w, 64, 32768, 1e-6, BF16, p, None) == E
    p = mk(_abi.KS_KERNEL_TWOPASS_ROW, 4, 256)
    assert _abi.ks_rms_norm_planned(a, b + 2, w, 64, 32768, 1e-6, BF16, p, None) == E  # unaligned


def test_split_two_pass_plans_are_checked():
    a, b, w = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    mk = _abi.make_plan
    for p in (mk(_abi.KS_KERNEL_TWOPASS_ROW, 4, 256, cluster=9),    # cluster over 8
              mk(_abi.KS_KERNEL_TWOPASS_ROW, 4, 256, 3, cluster=4),  # rows in flight: 1 or 2
              mk(_abi.KS_KERNEL_TWOPASS_ROW, 3, 256, cluster=4),    # unsupported vector count
              mk(_abi.KS_KERNEL_TWOPASS_ROW, 2, 2048, cluster=4)):  # block over 1024
        assert _abi.ks_rms_norm_planned(a, b, w, 64, 32768, 1e-6, BF16, p, None) == E
    # 8 CTAs over a row of 7 vectors: one would own none
    p = mk(_abi.KS_KERNEL_TWOPASS_ROW, 2, 32, cluster=8)
    assert _abi.ks_fused_add_rms_norm_planned(a, b, w, 64, 56, 1e-6, BF16, p, None) == E
    assert "without vectors" in _abi.ks_last_error()


def test_split_staged_plans_are_checked():
    a, b, w = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    mk = _abi.make_plan
    rows, hidden = 64, 32768  # 4096 vectors of bf16
    ok = mk(_abi.KS_KERNEL_BULK_ROW, 4, 512, 2, cluster=2)
    bad = [
        mk(_abi.KS_KERNEL_BULK_ROW, 4, 256, 2, cluster=2),   # 256 x 4 < the 2048-vector slice
        mk(_abi.KS_KERNEL_BULK_ROW, 4, 512, 2, cluster=9),   # cluster over 8
        mk(_abi.KS_KERNEL_BULK_ROW, 4, 512, 8, cluster=2),   # 8 x 32 KB > 226 KB
        mk(_abi.KS_KERNEL_BULK_ROW, 4, 512, 2, cluster=1),   # one CTA cannot hold 4096 vectors
    ]
    for p in bad:
        assert _abi.ks_rms_norm_planned(a, b, w, rows, hidden, 1e-6, BF16, p, None) == E
    # fused: two slices per stage, 4 x 64 KB does not fit
    p = mk(_abi.KS_KERNEL_BULK_ROW, 4, 512, 4, cluster=2)
    assert _abi.ks_fused_add_rms_norm_planned(a, b, w, rows, hidden, 1e-6, BF16, p, None) == E
    # a cluster so large that one of its CTAs would own no vector (8 CTAs, 7 vectors)
    p = mk(_abi.KS_KERNEL_BULK_ROW, 4, 32, 2, cluster=8)
    assert _abi.ks_rms_norm_planned(a, b, w, rows, 56, 1e-6, BF16, p, None) == E
    assert "without vectors" in _abi.ks_last_error()
    del ok


def test_planned_entry_points_reject_plans_that_do_not_fit():
    """Explicit plans are arguments: checked before any CUDA call."""
    a, b, w = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    mk = _abi.make_plan
    bad = [
        mk(_abi.KS_KERNEL_CTA_ROW, 4, 96),          # 96 threads x 4 vectors < 1024 vectors
        mk(_abi.KS_KERNEL_CTA_ROW, 4, 1024),        # over the 512-thread bound at 4 vectors
        mk(_abi.KS_KERNEL_CTA_ROW, 3, 512),         # unsupported vector count
        mk(_abi.KS_KERNEL_WARP_ROW, 4, 64),         # a warp cannot cover 1024 vectors
        mk(_abi.KS_KERNEL_WARP_ROW, 8, 64),         # nor at 8 vectors per lane (256)
        mk(_abi.KS_KERNEL_WARP_ROW, 3, 64),         # unsupported vector count
        mk(_abi.KS_KERNEL_BULK_ROW, 4, 256, 0),     # no stages
        mk(_abi.KS_KERNEL_BULK_ROW, 4, 256, 15),    # 15 x 16 KB > 227 KB
        mk(_abi.KS_KERNEL_SCALAR, 0, 48),           # not a multiple of 32
        mk(9, 4, 256),                              # unknown kernel
    ]
    for p in bad:
        assert _abi.ks_rms_norm_planned(a, b, w, 64, 8192, 1e-6, BF16, p, None) == E
    # warp-row teams: 8, 16 or 32 lanes, at most 4 vectors a lane below 32 (rows of 8 vectors)
    for team, v in ((4, 2), (12, 1), (24, 1), (8, 6), (16, 8)):
        p = mk(_abi.KS_KERNEL_WARP_ROW, v, 64, team=team)
        assert _abi.ks_rms_norm_planned(a, b, w, 64, 64, 1e-6, BF16, p, None) == E, (team, v)
    p = mk(_abi.KS_KERNEL_WARP_ROW, 1, 64, team=8)  # 8 lanes x 1 vector < 9 vectors
    assert _abi.ks_rms_norm_planned(a, b, w, 64, 72, 1e-6, BF16, p, None) == E
    # a vector plan on an unaligned pointer
    p = mk(_abi.KS_KERNEL_CTA_ROW, 4, 256)
    assert _abi.ks_rms_norm_planned(a, b + 2, w, 64, 8192, 1e-6, BF16, p, None) == E
    # fused rings hold two rows per stage: 8 x 32 KB does not fit
    p = mk(_abi.KS_KERNEL_BULK_ROW, 4, 256, 8)
    assert _abi.ks_fused_add_rms_norm_planned(a, b, w, 64, 8192, 1e-6, BF16, p, None) == E
    assert _abi.load().ks_rms_norm_planned(a, b, w, 64, 8192, 1e-6, BF16, None, None) == E


def test_host_chunk_rows():
    # plain: a slot (workspace / 3, rounded down to 256 bytes) of whole rows
    assert _abi.ks_host_chunk_rows(0, 8192, BF16, 3 * 16384 * 100) == 100
    # fused: x rows then residual rows at the next 256-byte boundary
    assert _abi.ks_host_chunk_rows(1, 8192, BF16, 3 * 16384 * 100) == 50
    # 200-byte rows in a 1024-byte slot: 2 fit (x at 0..400, residual at 512..912); 3 need 768 + 600
    assert _abi.ks_host_chunk_rows(1, 100, BF16, 3 * 1024) == 2
    assert _abi.ks_host_chunk_rows(0, 8192, BF16, 3 * 16383) == 0
    assert _abi.ks_host_chunk_rows(2, 8192, BF16, 1 << 20) == -1
    assert _abi.ks_host_chunk_rows(0, 8192, 9, 1 << 20) == -1


@pytest.mark.parametrize("fused", [False, True])
def test_host_entry_points_reject_invalid_arguments(fused):
    call = _abi.ks_fused_add_rms_norm_host if fused else _abi.ks_rms_norm_host
    a, b, w, ws = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    assert call(a, b, w, 4, 0, 1e-6, BF16, ws, 1 << 20, None) == E
    assert call(a, b, w, 4, 64, float("nan"), BF16, ws, 1 << 20, None) == E
    assert call(a, b, w, 4, 64, 1e-6, BF16, ws, 0, None) == E               # empty workspace
    assert call(a, b, w, 4, 8192, 1e-6, BF16, ws, 3 * 1000, None) == E      # no row fits a slot
    assert "holds no row" in _abi.ks_last_error()
    assert call(a, b, w, 4, 64, 1e-6, 7, ws, 1 << 20, None) == _abi.KS_ERR_UNSUPPORTED_DTYPE
    assert call(a, b, ws + 64, 4, 64, 1e-6, BF16, ws, 1 << 20, None) == _abi.KS_ERR_OVERLAP
    assert call(0, 0, 0, 0, 64, 1e-6, BF16, 0, 0, None) == _abi.KS_SUCCESS   # empty input


def test_launch_options():
    assert _abi.ks_get_launch_options() == 0  # off by default
    assert _abi.ks_set_launch_options(4) == _abi.KS_ERR_INVALID_ARGUMENT
    assert _abi.ks_set_launch_options(_abi.KS_LAUNCH_PDL) == _abi.KS_SUCCESS
    assert _abi.ks_get_launch_options() == _abi.KS_LAUNCH_PDL
    assert _abi.ks_set_launch_options(0) == _abi.KS_SUCCESS
    assert _abi.ks_get_launch_options() == 0


def test_planned_flags_validated():
    a, b, w = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    p = _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, 4, 256, flags=8)
    assert _abi.ks_rms_norm_planned(a, b, w, 64, 8192, 1e-6, BF16, p, None) == \
        _abi.KS_ERR_INVALID_ARGUMENT


def test_latency_regime_choices():
    # widest fused rows, few of them: a cluster of 8 CTAs per row, 1 vector per thread
    for hidden in (14336, 16384):
        p = plan(1, 7, hidden, bps=2)
        assert p.kernel == _abi.KS_KERNEL_CLUSTER_ROW and p.cluster == 8 and p.vec_per_thread == 1
        assert p.block * 8 * p.cluster >= hidden and p.grid == 7 * 8 and p.rows_per_pass == 7
        assert p.team == p.block * 8
    # too many rows for clusters of 8 on 152 SMs: the CTA kernel
    assert plan(1, 20, 16384).kernel == _abi.KS_KERNEL_CTA_ROW
    # narrower plain rows, few of them: 2 vectors per thread, twice the threads
    p = plan(0, 33, 4096)
    assert p.kernel == _abi.KS_KERNEL_CTA_ROW and p.vec_per_thread == 2 and p.block == 256
    # plain rows wider than 1024 vectors keep 4 vectors per thread
    p = plan(0, 33, 16384)
    assert p.kernel == _abi.KS_KERNEL_CTA_ROW and p.vec_per_thread == 4 and p.block == 512


@pytest.mark.parametrize("dtype,off", [(F32, 2), (F32, 1), (BF16, 1), (F16, 1)])
def test_pointers_not_aligned_to_the_element_are_rejected(dtype, off):
    """Every kernel accesses whole elements: a pointer that is not a multiple of the element size
    is an argument error for every entry point, found before any CUDA call."""
    E = _abi.KS_ERR_INVALID_ARGUMENT
    a, b, w, c = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30)
    rows, h = 8, 64
    for args in ((a + off, b, w), (a, b + off, w), (a, b, w + off)):
        assert _abi.ks_rms_norm(*args, rows, h, 1e-6, dtype, None) == E
        assert "aligned to the" in _abi.ks_last_error()
        assert _abi.ks_fused_add_rms_norm(*args, rows, h, 1e-6, dtype, None) == E
        p = _abi.make_plan(_abi.KS_KERNEL_SCALAR, 0, 64)
        assert _abi.ks_rms_norm_planned(*args, rows, h, 1e-6, dtype, p, None) == E
        assert _abi.ks_rms_norm_host(*args, rows, h, 1e-6, dtype, c, 1 << 24, None) == E
        assert _abi.ks_fused_add_rms_norm_host(*args, rows, h, 1e-6, dtype, c, 1 << 24, None) == E
        assert _abi.ks_fused_add_rms_norm_host_noalloc(*args, rows, h, 1e-6, dtype, None) == E
    assert _abi.ks_rms_norm_host(a, b, w, rows, h, 1e-6, dtype, c + off, 1 << 24, None) == E
    assert _abi.ks_silu_and_mul(a + off, b, rows, h, dtype, None) == E
    assert _abi.ks_silu_and_mul(a, b + off, rows, h, dtype, None) == E
    assert _abi.ks_softmax(a + off, b, rows, h, dtype, None) == E
    assert _abi.ks_softmax(a, b + off, rows, h, dtype, None) == E
    assert _abi.ks_layer_norm(a + off, b, w, c, rows, h, 1e-5, dtype, None) == E
    assert _abi.ks_layer_norm(a, b, w + off, None, rows, h, 1e-5, dtype, None) == E
    assert _abi.ks_layer_norm(a, b, None, c + off, rows, h, 1e-5, dtype, None) == E


@pytest.mark.parametrize("dtype", [BF16, F16, F32])
@pytest.mark.parametrize("op", [0, 1])
def test_every_width_gets_a_valid_plan(dtype, op):
    """Every row width from 1 to 2100 16-byte vectors (and an element more, which cannot be
    vectorised), at row counts around the heuristic's thresholds (SMs, 4 x SMs): the plan obeys
    the rules the planned entry points enforce, so the default path never builds a launch the
    library would refuse."""
    per = 4 if dtype == F32 else 8
    for rows in (1, 19, 152, 153, 607, 608, 65536):
        for hv in range(1, 2101):
            for hidden in (hv * per, hv * per + 1):
                p = plan(op, rows, hidden, dtype, bps=4)
                assert p.block % 32 == 0 and 32 <= p.block <= 1024, (rows, hidden, p.as_dict())
                assert p.grid >= 1
                if hidden % per:
                    assert p.kernel == _abi.KS_KERNEL_SCALAR
                    continue
                if p.kernel == WARP:
                    assert p.vec_per_thread in (1, 2, 4, 6, 8) and p.block <= 256
                    assert 32 * p.vec_per_thread >= hv, (rows, hidden)
                elif p.kernel == CTA:
                    assert p.vec_per_thread in (2, 4)
                    assert p.block <= (1024 if p.vec_per_thread == 2 else 512)
                    assert p.block * p.vec_per_thread >= hv, (rows, hidden)
                elif p.kernel == TWO:
                    assert p.vec_per_thread in (2, 4) and p.block <= 1024
                    if p.cluster >= 2:
                        slice_ = -(-hv // p.cluster)
                        assert p.cluster <= 8 and p.grid % p.cluster == 0
                        assert (p.cluster - 1) * slice_ < hv, (rows, hidden)
                elif p.kernel == BULK:
                    C = p.cluster if p.cluster >= 2 else 1
                    slice_ = -(-hv // C)
                    # the shared-memory rows kernel (plain op, split) runs up to 1024 threads
                    # at 4 vectors and needs 2 stages
                    smem_rows = bool(p.flags & _abi.KS_PLAN_SMEM_ROWS)
                    assert not smem_rows or (op == 0 and C >= 2 and p.stages >= 2)
                    bound = 1024 if smem_rows and p.vec_per_thread == 4 else 512
                    assert p.block <= bound and 1 <= p.stages <= 16 and C <= 8
                    assert p.vec_per_thread == 4 or (p.vec_per_thread == 8 and op == 0 and C >= 2)
                    assert p.block * p.vec_per_thread >= slice_ and (C - 1) * slice_ < hv
                    assert p.smem_bytes <= 226 * 1024 and p.grid % C == 0
                elif p.kernel == _abi.KS_KERNEL_CLUSTER_ROW:
                    assert 2 <= p.cluster <= 8 and p.grid % p.cluster == 0
                    assert p.vec_per_thread in (1, 2, 4) and p.block <= 512
                    slice_ = -(-hv // p.cluster)
                    assert p.block * p.vec_per_thread >= slice_ and (p.cluster - 1) * slice_ < hv
                else:
                    raise AssertionError(f"unexpected kernel {p.kernel} for {rows} x {hidden}")


# ------------------------------------------------------------- the next operators' launch plans

def op_plan(op, rows, hidden, dtype=BF16, aligned=True, sms=152):
    st, p = _abi.ks_plan_launch(op, rows, hidden, dtype, aligned, sms, 0)
    assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
    return p


def test_next_op_plans_follow_the_bands():
    """ks_plan_launch reports the next operators' plans: the width bands for many narrow rows,
    the general rules otherwise, the scalar kernel for rows that cannot be vectorised."""
    SM, LN, SW = _abi.OP_SOFTMAX, _abi.OP_LAYER_NORM, _abi.OP_SILU_AND_MUL
    # Softmax 16-bit: rows of 64..127 vectors take warp rows at 4 vectors a lane, prefetching
    p = op_plan(SM, 1000, 72 * 8)
    assert (p.kernel, p.vec_per_thread, p.block, p.flags) == (WARP, 4, 128, 0)
    # ... but not in the latency regime (rows <= SMs): a CTA per row
    assert op_plan(SM, 100, 72 * 8).kernel == CTA
    # Softmax fp32 rows of 193..208 vectors: CTA rows at 4 vectors without prefetch
    p = op_plan(SM, 1000, 200 * 4, F32)
    assert (p.kernel, p.vec_per_thread, p.flags) == (CTA, 4, _abi.KS_PLAN_NO_PREFETCH)
    assert p.block == 64
    # Softmax 16-bit rows of at most 16 vectors: teams of 8 lanes at 2 vectors, 4 rows a warp
    p = op_plan(SM, 1000, 16 * 8)
    assert (p.kernel, p.team, p.vec_per_thread, p.block) == (WARP, 8, 2, 128)
    # LayerNorm fp16 rows of 33..56 vectors: teams of 16 lanes at 4 vectors
    p = op_plan(LN, 1000, 40 * 8, F16)
    assert (p.kernel, p.team, p.vec_per_thread) == (WARP, 16, 4)
    # Softmax rows of 128..1024 vectors: CTA rows at 4 vectors without prefetch; wider prefetch
    p = op_plan(SM, 1000, 512 * 8)
    assert (p.kernel, p.vec_per_thread, p.block, p.flags) == (CTA, 4, 128, _abi.KS_PLAN_NO_PREFETCH)
    assert op_plan(SM, 1000, 1536 * 8).flags == 0
    # rows wider than 2048 vectors: the wide multi-pass kernel
    p = op_plan(SM, 1000, 4096 * 8)
    assert (p.kernel, p.vec_per_thread, p.block) == (TWO, 4, 256)
    # LayerNorm fp16 rows of 65..128 vectors: warp rows at 4 vectors
    p = op_plan(LN, 1000, 96 * 8, F16)
    assert (p.kernel, p.vec_per_thread, p.flags) == (WARP, 4, 0)
    # LayerNorm many rows of 1024 bf16 vectors: the staged ring; 1280: a 2-stage ring with the
    # weight and bias rows in shared memory; 2560: the wide kernel's 128 threads
    p = op_plan(LN, 32768, 1024 * 8)
    assert (p.kernel, p.vec_per_thread, p.block, p.stages, p.flags) == (BULK, 4, 256, 4, 0)
    p = op_plan(LN, 32768, 1280 * 8)
    assert (p.kernel, p.block, p.stages, p.flags) == (BULK, 320, 2, _abi.KS_PLAN_AFFINE_SMEM)
    p = op_plan(LN, 32768, 2560 * 8)
    assert (p.kernel, p.block) == (TWO, 128)
    # SwiGLU: the row kernel for rows of a multiple of 32 vectors (fp32: 64), else the flat walk
    # on 128-thread CTAs
    p = op_plan(SW, 1000, 1024 * 8)
    assert (p.kernel, p.block) == (CTA, 256)
    assert op_plan(SW, 1000, 64 * 8).kernel == CTA
    p = op_plan(SW, 1000, 65 * 8)
    assert (p.kernel, p.block) == (_abi.KS_KERNEL_FLAT, 128)
    assert op_plan(SW, 1000, 128 * 4, F32).kernel == CTA
    assert op_plan(SW, 1000, 96 * 4, F32).kernel == _abi.KS_KERNEL_FLAT
    # rows that cannot be vectorised
    for op in (SM, LN, SW):
        assert op_plan(op, 10, 1001).kernel == _abi.KS_KERNEL_SCALAR
        assert op_plan(op, 10, 1024, aligned=False).kernel == _abi.KS_KERNEL_SCALAR
    assert op_plan(SM, 0, 1024).kernel == _abi.KS_KERNEL_NONE


def test_affine_smem_flag_only_for_the_layer_norm_ring():
    """KS_PLAN_AFFINE_SMEM is refused on any plan but LayerNorm's staged ring, and a ring whose
    stages plus the weight and bias rows exceed shared memory is refused (before any CUDA call;
    every plan here is invalid, so the fake pointers are never used)."""
    E = _abi.KS_ERR_INVALID_ARGUMENT
    a, b, c = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    F = _abi.KS_PLAN_AFFINE_SMEM
    # RMSNorm: an unknown flag
    p = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 256, 2, flags=F)
    assert _abi.ks_rms_norm_planned(a, b, c, 64, 8192, 1e-6, BF16, p, None) == E
    # Softmax and LayerNorm CTA rows: not the ring
    p = _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, 4, 256, flags=F)
    assert _abi.ks_softmax_planned(a, b, 64, 8192, BF16, p, None) == E
    assert _abi.ks_layer_norm_planned(a, b, None, None, 64, 8192, 1e-5, BF16, p, None) == E
    # LayerNorm ring of 2048 vectors: 6 stages fit alone (192 KiB), not with two more rows
    p = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 512, 6, flags=F)
    assert _abi.ks_layer_norm_planned(a, b, None, None, 64, 16384, 1e-5, BF16, p, None) == E
    # rows of 2560 vectors: a 640-thread ring only with the flag; past 1024 threads never
    p = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 640, 2)
    assert _abi.ks_layer_norm_planned(a, b, None, None, 64, 20480, 1e-5, BF16, p, None) == E
    p = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 1056, 2, flags=F)
    assert _abi.ks_layer_norm_planned(a, b, None, None, 64, 33792, 1e-5, BF16, p, None) == E


def test_smem_rows_flag_only_for_the_plain_split_ring():
    """KS_PLAN_SMEM_ROWS is refused on the fused op, on a staged ring of one CTA per row or of
    one stage, and on any other kernel (before any CUDA call; every plan here is invalid, so the
    fake pointers are never used)."""
    E = _abi.KS_ERR_INVALID_ARGUMENT
    a, b, c = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    F = _abi.KS_PLAN_SMEM_ROWS
    good = _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 256, 2, flags=F, cluster=4)
    assert _abi.ks_fused_add_rms_norm_planned(a, b, c, 64, 32768, 1e-6, BF16, good, None) == E
    for p in (_abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 512, 2, flags=F),
              _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 256, 1, flags=F, cluster=4),
              _abi.make_plan(_abi.KS_KERNEL_TWOPASS_ROW, 4, 256, flags=F, cluster=4),
              _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, 4, 512, flags=F),
              # clusters past 8 CTAs only with the flag, and never past 16
              _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 128, 2, cluster=16),
              _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 128, 2, flags=F, cluster=17),
              # blocks past 512 threads only with the flag at 4 vectors, and never past 1024
              _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 1024, 2, cluster=2),
              _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 8, 1024, 2, flags=F, cluster=2),
              _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 1056, 2, flags=F, cluster=2)):
        assert _abi.ks_rms_norm_planned(a, b, c, 64, 32768, 1e-6, BF16, p, None) == E
    # the next operators take no such flag
    p = _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, 4, 256, flags=F)
    assert _abi.ks_softmax_planned(a, b, 64, 8192, BF16, p, None) == E


def test_next_op_planned_entry_points_check_the_plan():
    """Explicit plans for SwiGLU, Softmax and LayerNorm are arguments: checked before any CUDA
    call."""
    a, b = FAKE, FAKE + (1 << 30)
    E = _abi.KS_ERR_INVALID_ARGUMENT
    mk = _abi.make_plan
    NP = _abi.KS_PLAN_NO_PREFETCH
    rows, h = 64, 4096  # 512 bf16 vectors
    for p in (mk(WARP, 8, 128),                      # a warp covers 256 vectors, not 512
              mk(CTA, 4, 64),                        # 64 x 4 < 512
              mk(CTA, 2, 512, flags=NP),             # no CTA-row variant without prefetch at 2
              mk(CTA, 4, 1024),                      # block over 512
              mk(BULK, 4, 128, 2),                   # the ring is LayerNorm's
              mk(TWO, 2, 256),                       # the wide kernel steps 4 vectors
              mk(_abi.KS_KERNEL_FLAT, 2, 256),       # SwiGLU's
              mk(CTA, 4, 100),                       # not a multiple of 32
              mk(CTA, 4, 128, flags=8)):             # unknown flag
        assert _abi.ks_softmax_planned(a, b, rows, h, BF16, p, None) == E
    assert _abi.ks_softmax_planned(a, b + 2, rows, h, BF16, mk(CTA, 4, 128), None) == E  # unaligned
    for p in (mk(WARP, 4, 128, flags=NP),            # LayerNorm always prefetches
              mk(BULK, 4, 128, 1),                   # one stage
              mk(BULK, 4, 64, 2),                    # 64 x 4 < 512 vectors
              mk(TWO, 4, 1024)):                     # the LayerNorm wide kernel is bounded at 512
        assert _abi.ks_layer_norm_planned(a, b, None, None, rows, h, 1e-5, BF16, p, None) == E
    # a ring too large for shared memory: 8 stages of 2048 vectors (256 KiB)
    p = mk(BULK, 4, 512, 8)
    assert _abi.ks_layer_norm_planned(a, b, None, None, rows, 16384, 1e-5, BF16, p, None) == E
    for p in (mk(WARP, 4, 128), mk(_abi.KS_KERNEL_FLAT, 2, 512), mk(CTA, 2, 288)):
        assert _abi.ks_silu_and_mul_planned(a, b, rows, h, BF16, p, None) == E
    assert _abi.load().ks_softmax_planned(a, b, rows, h, BF16, None, None) == E


@pytest.mark.parametrize("dtype", [BF16, F16, F32])
def test_every_next_op_plan_is_a_valid_launch(dtype):
    """Row widths from 1 to 4400 vectors, few and many rows: each default plan of Softmax,
    LayerNorm and SwiGLU obeys the rules the planned entry points enforce (a team that covers the
    row, a block within the kernel's bound, a variant that exists), so the default path never
    builds a launch the library would refuse."""
    per = 4 if dtype == F32 else 8
    for rows in (7, 152, 153, 5000):
        for hv in list(range(1, 601)) + list(range(601, 4400, 7)):
            for op in (_abi.OP_SOFTMAX, _abi.OP_LAYER_NORM, _abi.OP_SILU_AND_MUL):
                p = op_plan(op, rows, hv * per, dtype)
                assert p.block % 32 == 0 and 32 <= p.block <= 1024, (op, rows, hv, p.as_dict())
                npf = bool(p.flags & _abi.KS_PLAN_NO_PREFETCH)
                if op == _abi.OP_SILU_AND_MUL:
                    assert p.kernel in (_abi.KS_KERNEL_FLAT, CTA) and p.block <= 256
                    continue
                if p.kernel == WARP:
                    assert p.team in (8, 16, 32) and p.block <= 128 and p.block % p.team == 0
                    assert p.vec_per_thread in ((2, 4, 6, 8) if p.team == 32 else (2, 4))
                    assert p.team * p.vec_per_thread >= hv, (op, rows, hv)
                    assert not (npf and op == _abi.OP_LAYER_NORM)
                elif p.kernel == CTA:
                    assert p.vec_per_thread in (1, 2, 4) and p.block <= 512
                    assert p.block * p.vec_per_thread >= hv, (op, rows, hv)
                    assert not npf or (op == _abi.OP_SOFTMAX and p.vec_per_thread == 4)
                elif p.kernel == BULK:
                    assert op == _abi.OP_LAYER_NORM and p.vec_per_thread == 4 and 2 <= p.stages <= 8
                    assert p.block * 4 >= hv and 128 + p.stages * hv * 16 <= 226 * 1024
                else:
                    assert p.kernel == TWO and p.vec_per_thread == 4
                    assert p.block <= (512 if op == _abi.OP_LAYER_NORM else 1024)
