"""Maximum sizes: tensors of more than 2^32 elements (8 GiB and more), where any 32-bit element or
byte offset would wrap. Every op runs at such a size through its default entry point; sampled
rows (first, last, middle, seeded others) are compared with the oracle, and the fused residual
is also checked on every row against the rounded sum computed independently by torch."""
import pytest
import torch

import oracle
import row_wise_rmsnorm_ks_gb300 as ks
from gpu_common import compare_output, sample_rows
from helpers import bits_equal
from row_wise_rmsnorm_ks_gb300 import synth

pytestmark = pytest.mark.gpu

ROWS, H = 262144, 16384  # 2^32 elements: 8 GiB per bf16 tensor


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _gib_free(device) -> float:
    free, _ = torch.cuda.mem_get_info(device)
    return free / 2**30


@pytest.fixture
def big(cuda_device):
    if _gib_free(cuda_device) < 48:
        pytest.skip("needs about 48 GiB of free device memory")
    yield cuda_device
    _free()


def _rows(x, idx):
    return x[idx.to(x.device)].cpu()


@pytest.mark.parametrize("rows", [ROWS, ROWS + 3])
def test_rms_norm_over_2_pow_32_elements(big, rows):
    x = synth.cast(synth.normal_dev((rows, H), synth.SEED_X, big), "bf16")
    w = synth.weight(H, "bf16").to(big)
    assert x.numel() >= 2**32
    y = ks.rms_norm(x, w, 1e-5)
    idx = sample_rows(rows, k=32)
    ref, _ = oracle.rms_norm(_rows(x, idx), w.cpu(), 1e-5)
    compare_output(_rows(y, idx), ref, torch.bfloat16, H, f"max size rms_norm [{rows},{H}]")


def test_fused_over_2_pow_32_elements(big):
    rows = ROWS + 1
    x = synth.cast(synth.normal_dev((rows, H), synth.SEED_X, big), "bf16")
    r = synth.cast(synth.normal_dev((rows, H), synth.SEED_RESIDUAL, big, std=2.0), "bf16")
    w = synth.weight(H, "bf16").to(big)
    idx = sample_rows(rows, k=32)
    x_host, r_host = _rows(x, idx), _rows(r, idx)
    expect_r = torch.empty_like(r)  # every row: the rounded sum, in chunks of rows
    for i in range(0, rows, 16384):
        expect_r[i:i + 16384] = (x[i:i + 16384].float() + r[i:i + 16384].float()).to(torch.bfloat16)
    ks.fused_add_rms_norm(x, r, w, 1e-5)
    for i in range(0, rows, 16384):
        assert bits_equal(r[i:i + 16384], expect_r[i:i + 16384]), f"residual rows {i}.."
    del expect_r
    ref_x, ref_r, _ = oracle.fused_add_rms_norm(x_host, r_host, w.cpu(), 1e-5)
    assert bits_equal(_rows(r, idx), ref_r)
    compare_output(_rows(x, idx), ref_x, torch.bfloat16, H, f"max size fused [{rows},{H}]")


def test_next_operators_over_2_pow_32_elements(big):
    rows = ROWS
    x = synth.cast(synth.normal_dev((rows, H), 21, big), "bf16")
    idx = sample_rows(rows, k=16)
    xs = _rows(x, idx)
    y = ks.softmax(x)
    ref, _ = oracle.softmax(xs)
    compare_output(_rows(y, idx), ref, torch.bfloat16, H, "max size softmax")
    del y
    _free()
    w = synth.weight(H, "bf16").to(big)
    b = synth.cast(synth.normal_np((H,), 22, std=0.1), "bf16").to(big)
    y = ks.layer_norm(x, w, b, 1e-5)
    ref, _ = oracle.layer_norm(xs, w.cpu(), b.cpu(), 1e-5)
    out = _rows(y, idx)
    away = ref.double().abs() > 0.05
    from helpers import tol_for, ulp_dist, within_tol
    assert int(ulp_dist(out[away], ref[away]).max()) <= 1
    assert within_tol(out, ref, *tol_for(torch.bfloat16, H))[0]
    del y
    _free()
    # SwiGLU over [rows/2, 2*H]: 2^32 input elements, the gate and up halves 2^31 apart
    g = x.view(rows // 2, 2 * H)
    y = ks.silu_and_mul(g)
    gi = sample_rows(rows // 2, k=16)
    ref, _ = oracle.silu_and_mul(_rows(g, gi))
    compare_output(_rows(y, gi), ref, torch.bfloat16, H, "max size silu_and_mul")
