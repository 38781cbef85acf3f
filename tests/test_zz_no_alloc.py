"""The allocation-free entry point, ks_fused_add_rms_norm_host_noalloc, called through the C ABI.

It serves callers that may not call cudaMalloc (device memory owned by another allocator, or
loops where an allocation would stall the device): it stages host rows through device scratch
built into the library instead of a workspace the caller lends. Two calls in a row must give the
same results as the existing entry point with a caller workspace, within the output tolerance the
other tests use, and the residual bit for bit; and, on its own, match the oracle (residual bit
for bit, output within the gate), also when two streams issue calls back to back over rows
that cycle through the scratch's three slots several times. This file is collected last.
"""
import pytest
import torch

import oracle
from gpu_common import compare_output
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


# rows that take 12 chunks, four cycles through the scratch's three 8 MiB slots
ORACLE_CASES = [(torch.bfloat16, 3000, 8192), (torch.float16, 3000, 8192),
                (torch.float32, 1500, 8192)]


@pytest.mark.parametrize("dtype,rows,hidden", ORACLE_CASES)
def test_noalloc_matches_oracle(cuda_device, dtype, rows, hidden):
    lib = _abi.load()
    w_host = synth.weight(hidden, dtype)
    w = w_host.to(cuda_device)
    x0, r0 = _inputs(rows, hidden, dtype, 231)
    ref_x, ref_r, _ = oracle.fused_add_rms_norm(x0, r0, w_host, 1e-6)
    x, r = x0.clone().pin_memory(), r0.clone().pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.ks_fused_add_rms_norm_host_noalloc(x.data_ptr(), r.data_ptr(), w.data_ptr(), rows,
                                                hidden, 1e-6, CODES[dtype], stream)
    assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
    torch.cuda.synchronize()
    assert bits_equal(r, ref_r), "residual differs from the oracle"
    compare_output(x, ref_x, dtype, hidden, f"noalloc vs oracle {dtype} [{rows},{hidden}]")


def test_noalloc_two_streams_back_to_back(cuda_device):
    """Two calls issued from two streams with no synchronisation between them, each over rows
    that cycle through the shared scratch several times: the library's pipeline streams order
    every reuse of a slot, so both results match the oracle."""
    lib = _abi.load()
    dtype, rows, hidden = torch.bfloat16, 3000, 8192
    w_host = synth.weight(hidden, dtype)
    w = w_host.to(cuda_device)
    sets = [_inputs(rows, hidden, dtype, seed) for seed in (241, 251)]
    refs = [oracle.fused_add_rms_norm(x0, r0, w_host, 1e-6)[:2] for x0, r0 in sets]
    bufs = [(x0.clone().pin_memory(), r0.clone().pin_memory()) for x0, r0 in sets]
    streams = [torch.cuda.Stream(cuda_device), torch.cuda.Stream(cuda_device)]
    torch.cuda.synchronize()
    for (x, r), s in zip(bufs, streams):
        st = lib.ks_fused_add_rms_norm_host_noalloc(x.data_ptr(), r.data_ptr(), w.data_ptr(), rows,
                                                    hidden, 1e-6, _abi.KS_DTYPE_BF16, s.cuda_stream)
        assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
    for s in streams:
        s.synchronize()
    for i, ((x, r), (ref_x, ref_r)) in enumerate(zip(bufs, refs)):
        assert bits_equal(r, ref_r), f"stream {i}: residual differs from the oracle"
        compare_output(x, ref_x, dtype, hidden, f"noalloc stream {i}")
