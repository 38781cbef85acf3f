"""The seeded input generators: deterministic, the stated laws, the stated special rows."""
import numpy as np
import torch

from row_wise_rmsnorm_ks_gb300 import synth


def test_deterministic():
    a = synth.normal_np((64, 128), 5)
    b = synth.normal_np((64, 128), 5)
    assert np.array_equal(a, b)
    # the first rows of a larger draw are the same draw (prefix property used by the CPU
    # reference arm of the bench)
    big = synth.normal_np((128, 128), 5)
    assert np.array_equal(big[:64], a)


def test_normal_law():
    a = synth.normal_np((1 << 20,), 1, std=2.0).astype(np.float64)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 2.0) < 0.01


def test_student_t3_law():
    a = synth.student_t3_np((1 << 20,), 2).astype(np.float64)
    # median 0, symmetric, heavy tails: P(|t3| > 5) = 0.0154
    assert abs(np.median(a)) < 0.01
    tail = np.mean(np.abs(a) > 5.0)
    assert 0.013 < tail < 0.018


def test_weight_law():
    w = synth.weight(1 << 16, torch.float32).double()
    assert abs(float(w.mean()) - 1.0) < 0.002 and abs(float(w.std()) - 0.1) < 0.002


def test_outlier_rows_count_and_range():
    for rows in (1, 7, 333, 65536):
        idx = synth.outlier_rows(rows)
        assert len(idx) == max(1, round(rows / 100))
        assert len(set(idx.tolist())) == len(idx) and idx.min() >= 0 and idx.max() < rows


def test_fp16_saturation():
    t = synth.cast(np.array([1e6, -1e6, 3.0], dtype=np.float32), torch.float16)
    assert t.tolist() == [65504.0, -65504.0, 3.0]
    assert torch.isfinite(synth.wide("fused_add_rms_norm", 1536, 7, "fp16").x.float()).all()


def test_medium_special_rows():
    w = synth.medium("bf16", rows=64, hidden=128)
    ci, zi = w.notes["const_row"], w.notes["zero_row"]
    assert ci != zi
    assert (w.x[zi].float() == 0).all()
    assert (w.x[ci].float() == w.x[ci, 0].float()).all() and float(w.x[ci, 0]) != 0


def test_wide_outliers_are_scaled():
    w = synth.wide("rms_norm", 1536, 333, "bf16")
    idx = w.notes["outlier_rows"]
    rms = w.x.float().pow(2).mean(dim=1).sqrt()
    others = [i for i in range(333) if i not in idx]
    assert float(rms[idx].min()) > 100 * float(rms[others].median())
