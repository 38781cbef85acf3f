"""Programmatic dependent launch: with KS_PLAN_PDL / KS_LAUNCH_PDL a row kernel may be scheduled
before the previous kernel in the stream finishes, and must wait for its writes before touching
memory. A chain of in-place launches, each reading what the one before wrote, must give the same
bits with and without it, for every kernel family."""
import pytest
import torch

import row_wise_rmsnorm_ks_gb300 as ks
from helpers import bits_equal
from row_wise_rmsnorm_ks_gb300 import _abi, synth

pytestmark = pytest.mark.gpu


def _chain(dev, rows, hidden, plan_flags, kernel, n=200):
    x = synth.cast(synth.normal_np((rows, hidden), 301), torch.bfloat16).to(dev)
    r = synth.cast(synth.normal_np((rows, hidden), 302), torch.bfloat16).to(dev)
    y = torch.empty_like(x)
    w = synth.weight(hidden, torch.bfloat16).to(dev)
    s = torch.cuda.current_stream().cuda_stream
    p = kernel(plan_flags)
    for _ in range(n):
        _abi.check(_abi.ks_fused_add_rms_norm_planned(x.data_ptr(), r.data_ptr(), w.data_ptr(),
                                                      rows, hidden, 1e-6, _abi.KS_DTYPE_BF16, p, s))
        _abi.check(_abi.ks_rms_norm_planned(y.data_ptr(), x.data_ptr(), w.data_ptr(), rows, hidden,
                                            1e-6, _abi.KS_DTYPE_BF16, p, s))
        _abi.check(_abi.ks_rms_norm_planned(x.data_ptr(), y.data_ptr(), w.data_ptr(), rows, hidden,
                                            1e-6, _abi.KS_DTYPE_BF16, p, s))
    torch.cuda.synchronize()
    return x.cpu(), r.cpu()


KERNELS = {
    "warp_row": lambda f: _abi.make_plan(_abi.KS_KERNEL_WARP_ROW, 4, 128, flags=f),
    "cta_row": lambda f: _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, 4, 64, flags=f),
    "cta_row_np": lambda f: _abi.make_plan(_abi.KS_KERNEL_CTA_ROW, 4, 64,
                                           flags=f | _abi.KS_PLAN_NO_PREFETCH),
    "bulk_row": lambda f: _abi.make_plan(_abi.KS_KERNEL_BULK_ROW, 4, 64, stages=2, flags=f),
    "scalar": lambda f: _abi.make_plan(_abi.KS_KERNEL_SCALAR, 0, 128, flags=f),
    "cluster_row": lambda f: _abi.make_plan(_abi.KS_KERNEL_CLUSTER_ROW, 2, 32, flags=f,
                                            cluster=4),
}


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("rows,hidden", [(4, 1536), (300, 1024)])
def test_pdl_chain_matches_plain_launches(cuda_device, kernel, rows, hidden):
    if kernel == "warp_row" and hidden > 1024:
        pytest.skip("a warp row holds at most 1024 bf16")
    ref = _chain(cuda_device, rows, hidden, 0, KERNELS[kernel])
    got = _chain(cuda_device, rows, hidden, _abi.KS_PLAN_PDL, KERNELS[kernel])
    assert bits_equal(got[0], ref[0]) and bits_equal(got[1], ref[1])


def test_process_wide_pdl_option(cuda_device):
    rows, hidden = 4, 1536
    x0 = synth.cast(synth.normal_np((rows, hidden), 303), torch.bfloat16)
    r0 = synth.cast(synth.normal_np((rows, hidden), 304), torch.bfloat16)
    w = synth.weight(hidden, torch.bfloat16).to(cuda_device)

    def run():
        x, r = x0.to(cuda_device), r0.to(cuda_device)
        for _ in range(300):
            ks.fused_add_rms_norm(x, r, w)
        torch.cuda.synchronize()
        return x.cpu(), r.cpu()

    ref = run()
    assert _abi.ks_set_launch_options(_abi.KS_LAUNCH_PDL) == _abi.KS_SUCCESS
    try:
        got = run()
    finally:
        _abi.ks_set_launch_options(0)
    assert bits_equal(got[0], ref[0]) and bits_equal(got[1], ref[1])
