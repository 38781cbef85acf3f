"""The allocation-free entry point, ks_fused_add_rms_norm_host_noalloc, called through the C ABI.

It serves callers that may not call cudaMalloc (device memory owned by another allocator, or
loops where an allocation would stall the device): it stages host rows through device scratch
built into the library instead of a workspace the caller lends. Two calls in a row must give the
same results as the existing entry point with a caller workspace, within the output tolerance the
other tests use, and the residual bit for bit. This file is collected last.
"""
import pytest
import torch

from helpers import bits_equal, tol_for, ulp_dist, within_tol
from row_wise_rmsnorm_ks_gb300 import _abi, synth

pytestmark = pytest.mark.gpu

CODES = {torch.bfloat16: _abi.KS_DTYPE_BF16, torch.float16: _abi.KS_DTYPE_F16,
         torch.float32: _abi.KS_DTYPE_F32}


def _inputs(rows, hidden, dtype, seed):
    x = synth.cast(synth.normal_np((rows, hidden), seed), dtype).pin_memory()
    r = synth.cast(synth.normal_np((rows, hidden), seed + 1, std=2.0), dtype).pin_memory()
    return x, r


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("rows,hidden", [(3000, 4096), (333, 8192), (17, 1001)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, dtype, rows, hidden):
    lib = _abi.load()
    w = synth.weight(hidden, dtype).to(cuda_device)
    e = torch.tensor([], dtype=dtype).element_size()
    ws = torch.empty(3 * (2 * 64 * hidden * e + 512), dtype=torch.uint8, device=cuda_device)
    stream = torch.cuda.current_stream().cuda_stream
    # the existing entry point (caller workspace) and the new one, each twice in a row
    xa, ra = _inputs(rows, hidden, dtype, 211)
    xb, rb = xa.clone().pin_memory(), ra.clone().pin_memory()
    for call in range(2):
        st = lib.ks_fused_add_rms_norm_host(xa.data_ptr(), ra.data_ptr(), w.data_ptr(), rows, hidden,
                                            1e-6, CODES[dtype], ws.data_ptr(), ws.numel(), stream)
        assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
        st = lib.ks_fused_add_rms_norm_host_noalloc(xb.data_ptr(), rb.data_ptr(), w.data_ptr(), rows,
                                                    hidden, 1e-6, CODES[dtype], stream)
        assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
        torch.cuda.synchronize()
        assert bits_equal(rb, ra), f"call {call}: residual differs"
        rtol, atol = tol_for(dtype, hidden)
        ok, worst, _ = within_tol(xb, xa, rtol, atol)
        assert ok, f"call {call}: normalised output beyond tolerance by {worst}"
        if dtype != torch.float32:
            assert int(ulp_dist(xb, xa).max()) <= 1
        # the next call starts both paths from the same rows (the scratch still holds this
        # call's chunks): its results must again agree
        xb.copy_(xa)
        rb.copy_(ra)


def test_noalloc_rejects_rows_wider_than_its_scratch(cuda_device):
    lib = _abi.load()
    w = torch.empty(8, dtype=torch.bfloat16, device=cuda_device)
    x = torch.empty(8, dtype=torch.bfloat16).pin_memory()
    r = torch.empty(8, dtype=torch.bfloat16).pin_memory()
    hidden = 4 << 20  # 8 MiB per row per tensor: two rows exceed an 8 MiB slot
    st = lib.ks_fused_add_rms_norm_host_noalloc(x.data_ptr(), r.data_ptr(), w.data_ptr(), 1,
                                                hidden, 1e-6, _abi.KS_DTYPE_BF16, None)
    assert st == _abi.KS_ERR_INVALID_ARGUMENT
    assert "built-in scratch" in _abi.ks_last_error()
