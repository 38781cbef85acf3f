"""GPU parity of the RMSNorm row kernel with several rows per warp (8- and 16-lane teams) and a
warp per row, through the explicit-plan entry points, against the oracle element by element.

A warp of 8- or 16-lane teams holds consecutive rows and runs as long as its first row does; its
teams past the last row must store nothing. So the cases take ragged row counts (not a multiple
of the rows a CTA holds), a small grid cap (every team walks many rows, the last pass partial),
widths that leave lanes of a team idle, and guard rows after the output that must stay untouched.
"""
import pytest
import torch

import oracle
from gpu_common import compare_output
from helpers import bits_equal
from row_wise_rmsnorm_ks_gb300 import _abi as A
from row_wise_rmsnorm_ks_gb300 import synth

pytestmark = pytest.mark.gpu
CODES = {torch.bfloat16: A.KS_DTYPE_BF16, torch.float16: A.KS_DTYPE_F16,
         torch.float32: A.KS_DTYPE_F32}
NP = A.KS_PLAN_NO_PREFETCH

# (rows, block, grid cap): one row; a few rows in one CTA; ragged counts over several CTAs with
# the grid the library sizes; ragged counts on 3 CTAs, so each team walks many rows
LAUNCHES = [(1, 32, 0), (5, 96, 0), (1001, 96, 0), (333, 256, 0), (1001, 256, 3), (77, 64, 2)]
GUARD = 3  # rows after the output that no launch may write


def _widths(dt):
    # row widths in 16-byte vectors: 1, 2, 3, 5, 8, 15, 16, 17, 31, 32, 33, 48, 64, 100, 128
    per = 4 if dt == torch.float32 else 8
    return [hv * per for hv in (1, 2, 3, 5, 8, 15, 16, 17, 31, 32, 33, 48, 64, 100, 128)]


@pytest.mark.parametrize("team", [8, 16, 32])
@pytest.mark.parametrize("v", [1, 2, 4])
@pytest.mark.parametrize("prefetch", [True, False], ids=["prefetch", "no_prefetch"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("op", ["rms_norm", "fused_add_rms_norm"])
def test_team_rows_match_oracle(cuda_device, team, v, prefetch, dtype, op):
    dt = synth.dtype_of(dtype)
    code = CODES[dt]
    s = torch.cuda.current_stream().cuda_stream
    per = 4 if dt == torch.float32 else 8
    ran = 0
    for hidden in _widths(dt):
        hv = hidden // per
        if team * v < hv:
            continue  # the team does not cover the row
        wt = synth.weight(hidden, dt)
        wd = wt.to(cuda_device)
        for rows, block, grid in LAUNCHES:
            plan = A.make_plan(A.KS_KERNEL_WARP_ROW, v, block, grid=grid,
                               flags=0 if prefetch else NP, team=team)
            seed = 600 + hv * 7 + rows
            x = synth.cast(synth.normal_np((rows + GUARD, hidden), seed, std=2.0), dt)
            xd = x.to(cuda_device)
            name = f"{op} {dtype} team {team} v{v} {'pf' if prefetch else 'np'} [{rows},{hidden}] b{block} g{grid}"
            if op == "rms_norm":
                yd = torch.full_like(xd, 7.0)
                A.check(A.ks_rms_norm_planned(yd.data_ptr(), xd.data_ptr(), wd.data_ptr(), rows,
                                              hidden, 1e-6, code, plan, s))
                ref, _ = oracle.rms_norm(x[:rows], wt, 1e-6)
                out = yd.cpu()
                compare_output(out[:rows], ref, dt, hidden, name)
                assert bool((out[rows:] == 7.0).all()), f"{name}: wrote past the last row"
            else:
                r = synth.cast(synth.normal_np((rows + GUARD, hidden), seed + 1), dt)
                rd = r.to(cuda_device)
                A.check(A.ks_fused_add_rms_norm_planned(xd.data_ptr(), rd.data_ptr(),
                                                        wd.data_ptr(), rows, hidden, 1e-6, code,
                                                        plan, s))
                ref_x, ref_r, _ = oracle.fused_add_rms_norm(x[:rows], r[:rows], wt, 1e-6)
                ox, orr = xd.cpu(), rd.cpu()
                assert bits_equal(orr[:rows], ref_r), name
                compare_output(ox[:rows], ref_x, dt, hidden, name)
                assert bits_equal(ox[rows:], x[rows:]) and bits_equal(orr[rows:], r[rows:]), \
                    f"{name}: wrote past the last row"
            ran += 1
    assert ran > 0
    st, flags = A.ks_device_faults(clear=True)
    assert st == A.KS_SUCCESS and flags == 0


def test_team_plans_are_checked(cuda_device):
    """A team of a size other than 8, 16 or 32 lanes, more than 4 vectors a lane on a sub-warp
    team, or a team that does not cover the row: refused before any launch."""
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device=cuda_device)
    w = torch.ones(64, dtype=torch.bfloat16, device=cuda_device)
    s = torch.cuda.current_stream().cuda_stream
    for team, v in ((4, 2), (12, 1), (8, 6), (16, 8)):
        p = A.make_plan(A.KS_KERNEL_WARP_ROW, v, 64, team=team)
        assert A.ks_rms_norm_planned(x.data_ptr(), x.data_ptr(), w.data_ptr(), 4, 64, 1e-6,
                                     A.KS_DTYPE_BF16, p, s) == A.KS_ERR_INVALID_ARGUMENT
    p = A.make_plan(A.KS_KERNEL_WARP_ROW, 1, 64, team=8)  # 8 lanes x 1 vector < 8 + 1 vectors
    x2 = torch.zeros((4, 72), dtype=torch.bfloat16, device=cuda_device)
    w2 = torch.ones(72, dtype=torch.bfloat16, device=cuda_device)
    assert A.ks_rms_norm_planned(x2.data_ptr(), x2.data_ptr(), w2.data_ptr(), 4, 72, 1e-6,
                                 A.KS_DTYPE_BF16, p, s) == A.KS_ERR_INVALID_ARGUMENT
