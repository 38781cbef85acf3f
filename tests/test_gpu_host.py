"""GPU parity of the host-buffer entry points (ks_rms_norm_host, ks_fused_add_rms_norm_host):
rows in host memory go through the device in chunks and come back. The residual must equal the
device-pointer path and the oracle bit for bit; the normalised output must meet the oracle's
output gate and stay within 1 ulp of the device path (a chunk may take another launch shape
than the whole batch, and the reduction order follows the launch shape)."""
import pytest
import torch

import oracle
import row_wise_rmsnorm_ks_gb300 as ks
from gpu_common import compare_output
from helpers import bits_equal, ulp_dist
from row_wise_rmsnorm_ks_gb300 import _abi, synth

pytestmark = pytest.mark.gpu


def _workspace(dev, nbytes):
    return torch.empty(nbytes, dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,hidden,ws_rows", [(1000, 4096, 64), (333, 1536, 7), (100, 8192, 1),
                                                 (77, 1001, 5), (5, 16384, 100)])
def test_host_plain(cuda_device, pinned, dtype, rows, hidden, ws_rows):
    dt = synth.dtype_of(dtype)
    e = torch.tensor([], dtype=dt).element_size()
    x = synth.cast(synth.normal_np((rows, hidden), 101), dt)
    if pinned:
        x = x.pin_memory()
    w = synth.weight(hidden, dt)
    ws = _workspace(cuda_device, 3 * ws_rows * hidden * e + 3 * 256)
    assert _abi.ks_host_chunk_rows(0, hidden, synth_code(dt), ws.numel()) >= ws_rows
    y = ks.rms_norm_host(x, w.to(cuda_device), 1e-6, workspace=ws)
    torch.cuda.synchronize()
    y_dev = ks.rms_norm(x.to(cuda_device), w.to(cuda_device), 1e-6).cpu()
    if dt != torch.float32:
        assert int(ulp_dist(y, y_dev).max()) <= 1
    ref, _ = oracle.rms_norm(x, w, 1e-6)
    compare_output(y, ref, dt, hidden, f"host rms_norm {dtype} [{rows},{hidden}] chunk {ws_rows}")


def synth_code(dt):
    return {torch.bfloat16: _abi.KS_DTYPE_BF16, torch.float16: _abi.KS_DTYPE_F16,
            torch.float32: _abi.KS_DTYPE_F32}[dt]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,hidden,ws_rows", [(1000, 4096, 64), (333, 1536, 7), (100, 8192, 1),
                                                 (77, 1001, 5), (5, 16384, 100)])
def test_host_fused(cuda_device, pinned, dtype, rows, hidden, ws_rows):
    dt = synth.dtype_of(dtype)
    e = torch.tensor([], dtype=dt).element_size()
    x = synth.cast(synth.normal_np((rows, hidden), 102), dt)
    r = synth.cast(synth.normal_np((rows, hidden), 103, std=2.0), dt)
    if pinned:
        x, r = x.pin_memory(), r.pin_memory()
    w = synth.weight(hidden, dt)
    ref_x, ref_r, _ = oracle.fused_add_rms_norm(x, r, w, 1e-6)
    xd, rd = x.to(cuda_device), r.to(cuda_device)
    ks.fused_add_rms_norm(xd, rd, w.to(cuda_device), 1e-6)
    ws = _workspace(cuda_device, 3 * (2 * ws_rows * hidden * e + 512))
    ks.fused_add_rms_norm_host(x, r, w.to(cuda_device), 1e-6, workspace=ws)
    torch.cuda.synchronize()
    assert bits_equal(r, rd.cpu()) and bits_equal(r, ref_r)
    if dt != torch.float32:
        assert int(ulp_dist(x, xd.cpu()).max()) <= 1
    compare_output(x, ref_x, dt, hidden, f"host fused {dtype} [{rows},{hidden}] chunk {ws_rows}")


def test_host_in_place_and_stream_order(cuda_device):
    """out == x on the host; a second call on the same stream and workspace reads the first
    call's results (calls sharing a workspace are ordered on one stream). The first pass is
    checked against the oracle from the pristine input; the composition against the device
    path bit for bit (the oracle never takes a GPU output as its input)."""
    rows, hidden = 4000, 2048  # 25 whole chunks of 160 rows
    x0 = synth.cast(synth.normal_np((rows, hidden), 104), torch.bfloat16)
    w = synth.weight(hidden, torch.bfloat16)
    ref1, _ = oracle.rms_norm(x0, w, 1e-6)
    # 160-row chunks: more rows than SMs, so each chunk takes the same launch shape as the whole
    # 4000-row batch on the device, and the bits must match exactly
    ws = _workspace(cuda_device, 3 * 160 * hidden * 2)
    assert _abi.ks_host_chunk_rows(0, hidden, _abi.KS_DTYPE_BF16, ws.numel()) == 160
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    st, p_chunk = _abi.ks_plan_launch(0, 160, hidden, _abi.KS_DTYPE_BF16, True, sms, 0)
    st, p_all = _abi.ks_plan_launch(0, rows, hidden, _abi.KS_DTYPE_BF16, True, sms, 0)
    assert (p_chunk.kernel, p_chunk.vec_per_thread, p_chunk.block, p_chunk.flags) == \
        (p_all.kernel, p_all.vec_per_thread, p_all.block, p_all.flags)
    wd = w.to(cuda_device)
    x = x0.clone().pin_memory()
    ks.rms_norm_host(x, wd, 1e-6, workspace=ws, out=x)
    torch.cuda.synchronize()
    compare_output(x, ref1, torch.bfloat16, hidden, "host in place, first pass")
    ks.rms_norm_host(x, wd, 1e-6, workspace=ws, out=x)
    ks.rms_norm_host(x, wd, 1e-6, workspace=ws, out=x)
    torch.cuda.synchronize()
    xd = x0.to(cuda_device)
    for _ in range(3):
        ks.rms_norm(xd, wd, 1e-6, out=xd)
    assert bits_equal(x, xd.cpu())


def test_host_side_stream(cuda_device):
    rows, hidden = 2000, 4096
    x = synth.cast(synth.normal_np((rows, hidden), 105), torch.bfloat16).pin_memory()
    r = synth.cast(synth.normal_np((rows, hidden), 106), torch.bfloat16).pin_memory()
    w = synth.weight(hidden, torch.bfloat16)
    ref_x, ref_r, _ = oracle.fused_add_rms_norm(x, r, w, 1e-6)
    ws = _workspace(cuda_device, 3 * 2 * 100 * hidden * 2 + 1024)
    s = torch.cuda.Stream()
    wd = w.to(cuda_device)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ks.fused_add_rms_norm_host(x, r, wd, 1e-6, workspace=ws)
    s.synchronize()
    assert bits_equal(r, ref_r)
    compare_output(x, ref_x, torch.bfloat16, hidden, "host fused side stream")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("rows,hidden", [(1000, 4096), (333, 1536), (77, 1001), (5, 16384)])
def test_host_direct_mode(cuda_device, dtype, rows, hidden):
    """No workspace: the kernels read and write pinned host rows over the host link."""
    dt = synth.dtype_of(dtype)
    x = synth.cast(synth.normal_np((rows, hidden), 107), dt).pin_memory()
    r = synth.cast(synth.normal_np((rows, hidden), 108, std=2.0), dt).pin_memory()
    w = synth.weight(hidden, dt)
    wd = w.to(cuda_device)
    ref_y, _ = oracle.rms_norm(x, w, 1e-6)
    ref_x, ref_r, _ = oracle.fused_add_rms_norm(x, r, w, 1e-6)
    y = ks.rms_norm_host(x, wd, 1e-6)
    torch.cuda.synchronize()
    assert y.is_pinned()
    compare_output(y, ref_y, dt, hidden, f"host direct rms_norm {dtype} [{rows},{hidden}]")
    ks.fused_add_rms_norm_host(x, r, wd, 1e-6)
    torch.cuda.synchronize()
    assert bits_equal(r, ref_r)
    compare_output(x, ref_x, dt, hidden, f"host direct fused {dtype} [{rows},{hidden}]")


def test_host_direct_mode_refuses_pageable_memory(cuda_device):
    """Pageable host memory is not mapped: the call is refused before any launch."""
    x = synth.cast(synth.normal_np((16, 1024), 109), torch.bfloat16)   # not pinned
    y = torch.empty_like(x)
    wd = synth.weight(1024, torch.bfloat16).to(cuda_device)
    st = _abi.ks_rms_norm_host(y.data_ptr(), x.data_ptr(), wd.data_ptr(), 16, 1024, 1e-6,
                               _abi.KS_DTYPE_BF16, None, 0, None)
    assert st == _abi.KS_ERR_INVALID_ARGUMENT and "page-locked" in _abi.ks_last_error()
    # a pinned input with a pageable output is refused too
    xp = x.pin_memory()
    st = _abi.ks_rms_norm_host(y.data_ptr(), xp.data_ptr(), wd.data_ptr(), 16, 1024, 1e-6,
                               _abi.KS_DTYPE_BF16, None, 0, None)
    assert st == _abi.KS_ERR_INVALID_ARGUMENT
    st, flags = _abi.ks_device_faults(clear=False)
    assert st == _abi.KS_SUCCESS and flags == 0
