"""GPU parity of the staged kernel that keeps each row slice in shared memory through both passes
(plan flag KS_PLAN_SMEM_ROWS), through the explicit-plan entry point, against the oracle element
by element.

The kernel keeps two rows in flight per cluster: iteration j forms row j's sum and sends it while
row j - 1 is written, and the sum slots cycle over four rows. So the cases take clusters with 1,
2, 3 and many rows (the pipeline's fill and drain, and slots reused many times), ragged slices
(the last CTA of a cluster with fewer vectors), rings of 2 to 6 stages, both weight widths, and
guard rows after the output that no launch may write. Clusters of more than 8 CTAs are a
non-portable size: where the device cannot place one, the call fails before any launch and the
case is skipped.
"""
import pytest
import torch

import oracle
from gpu_common import compare_output
from row_wise_rmsnorm_ks_gb300 import _abi as A
from row_wise_rmsnorm_ks_gb300 import synth

pytestmark = pytest.mark.gpu
CODES = {torch.bfloat16: A.KS_DTYPE_BF16, torch.float16: A.KS_DTYPE_F16,
         torch.float32: A.KS_DTYPE_F32}
GUARD = 3
# (cluster, stages, vectors of weight per thread)
SHAPES = [(2, 2, 4), (3, 3, 8), (8, 5, 4), (8, 2, 8), (4, 6, 8), (16, 3, 4), (16, 2, 8),
          (12, 4, 8), (2, 3, 4), (8, 3, 4)]
# (rows, clusters launched): one, two, three rows on one cluster; ragged counts over two and
# three clusters, so each cluster walks many rows
LAUNCHES = [(1, 1), (2, 1), (3, 1), (5, 2), (33, 2), (1001, 3)]


def _plan(hv, c, stages, v, clusters):
    # the block fitted to the slice: up to 1024 threads at 4 vectors of weight, 512 at 8 (at
    # hv 4100 and 24576 the shapes c2 and c8 at 4 vectors take 544 and 768 threads)
    slice_ = -(-hv // c)
    block = max(32, -(-(-(-slice_ // v)) // 32) * 32)
    if block > (1024 if v == 4 else 512) or (c - 1) * slice_ >= hv or \
            128 + stages * slice_ * 16 > 226 * 1024:
        return None
    return A.make_plan(A.KS_KERNEL_BULK_ROW, v, block, stages, grid=clusters * c,
                       flags=A.KS_PLAN_SMEM_ROWS, cluster=c)


@pytest.mark.parametrize("shape", SHAPES, ids=[f"c{c}s{s}v{v}" for c, s, v in SHAPES])
@pytest.mark.parametrize("hv", [1100, 4100, 24576])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_smem_rows_match_oracle(cuda_device, shape, hv, dtype):
    c, stages, v = shape
    dt = synth.dtype_of(dtype)
    per = 4 if dt == torch.float32 else 8
    hidden = hv * per
    code = CODES[dt]
    s = torch.cuda.current_stream().cuda_stream
    wt = synth.weight(hidden, dt)
    wd = wt.to(cuda_device)
    ran = 0
    for rows, clusters in LAUNCHES:
        if hv == 24576 and rows > 33:
            continue  # the oracle's time: the widest rows take the short launches only
        plan = _plan(hv, c, stages, v, clusters)
        if plan is None:
            continue
        x = synth.cast(synth.normal_np((rows + GUARD, hidden), 700 + rows + hv, std=2.0), dt)
        xd = x.to(cuda_device)
        yd = torch.full_like(xd, 7.0)
        st = A.ks_rms_norm_planned(yd.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows, hidden,
                                   1e-6, code, plan, s)
        if st == A.KS_ERR_CUDA and c > 8 and "resident" in A.ks_last_error():
            pytest.skip(f"the device places no cluster of {c}: {A.ks_last_error()}")
        A.check(st)
        ref, _ = oracle.rms_norm(x[:rows], wt, 1e-6)
        out = yd.cpu()
        name = f"smem rows {dtype} c{c} s{stages} v{v} [{rows},{hidden}] on {clusters} clusters"
        compare_output(out[:rows], ref, dt, hidden, name)
        assert bool((out[rows:] == 7.0).all()), f"{name}: wrote past the last row"
        ran += 1
    if ran == 0:
        pytest.skip("no launch of this shape fits the width")
    st, flags = A.ks_device_faults(clear=True)
    assert st == A.KS_SUCCESS and flags == 0


def test_smem_rows_plans_are_checked(cuda_device):
    """The flag on the fused op, on one CTA per row, on a ring of one stage, or beside a weight
    slice the threads do not cover: refused before any launch."""
    hv, c = 4096, 4
    x = torch.zeros((8, hv * 8), dtype=torch.bfloat16, device=cuda_device)
    r = torch.zeros_like(x)
    w = torch.ones(hv * 8, dtype=torch.bfloat16, device=cuda_device)
    s = torch.cuda.current_stream().cuda_stream
    F, E = A.KS_PLAN_SMEM_ROWS, A.KS_ERR_INVALID_ARGUMENT
    ok = A.make_plan(A.KS_KERNEL_BULK_ROW, 4, 256, 2, flags=F, cluster=c)
    assert A.ks_fused_add_rms_norm_planned(x.data_ptr(), r.data_ptr(), w.data_ptr(), 8, hv * 8,
                                           1e-6, A.KS_DTYPE_BF16, ok, s) == E
    for p in (A.make_plan(A.KS_KERNEL_BULK_ROW, 4, 512, 2, flags=F),
              A.make_plan(A.KS_KERNEL_BULK_ROW, 4, 256, 1, flags=F, cluster=c),
              A.make_plan(A.KS_KERNEL_BULK_ROW, 4, 128, 2, flags=F, cluster=c),
              A.make_plan(A.KS_KERNEL_CTA_ROW, 4, 512, flags=F)):
        assert A.ks_rms_norm_planned(x.data_ptr(), x.data_ptr(), w.data_ptr(), 8, hv * 8, 1e-6,
                                     A.KS_DTYPE_BF16, p, s) == E
