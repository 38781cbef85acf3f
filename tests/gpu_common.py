"""Helpers for the GPU parity tests: run a workload through the C ABI, run the oracle on the
same inputs (all rows, or sampled rows for the multi-gigabyte cases), compare."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
import row_wise_rmsnorm_ks_gb300 as ks
from helpers import bits_equal, tol_for, ulp_dist, within_tol
from row_wise_rmsnorm_ks_gb300 import synth

REPORT = os.environ.get("KS_PARITY_REPORT")


def record(name: str, **kv):
    """Append one parity result line when KS_PARITY_REPORT names a file."""
    if REPORT:
        with open(REPORT, "a") as f:
            f.write(json.dumps({"case": name, **kv}) + "\n")


def compare_output(out: torch.Tensor, ref: torch.Tensor, dtype, hidden: int, name: str):
    """The output gate: within the stated tolerance and, for 16-bit outputs, within 1 ulp."""
    rtol, atol = tol_for(dtype, hidden)
    ok, worst, idx = within_tol(out, ref, rtol, atol)
    ulps = int(ulp_dist(out, ref).max()) if out.numel() else 0
    n_diff = int((ulp_dist(out, ref) > 0).sum()) if out.numel() else 0
    record(name, max_ulp=ulps, worst_excess=worst, n=out.numel(), n_differ=n_diff)
    assert ok, f"{name}: tolerance exceeded by {worst} at flat index {idx}"
    if dtype != torch.float32:
        assert ulps <= 1, f"{name}: {ulps} ulp apart"
    return ulps


def sample_rows(rows: int, extra=(), k: int = 24, seed: int = 77) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    pick = {0, 1, 2, rows - 1, rows - 2, rows // 2}
    pick.update(int(i) for i in rng.choice(rows, size=min(k, rows), replace=False))
    pick.update(int(i) for i in extra)
    return torch.tensor(sorted(i for i in pick if 0 <= i < rows), dtype=torch.long)


def run_and_check(w: synth.Workload, device, rows_idx: torch.Tensor | None = None,
                  name: str | None = None):
    """Run workload `w` through the C ABI on `device` and compare with the oracle, on all rows
    or on rows_idx. Returns a dict of the device outputs (on the device)."""
    name = name or w.name
    x = w.x.to(device, copy=True)
    wt = w.weight.to(device)
    x_host = w.x.cpu() if rows_idx is None else w.x[rows_idx.to(w.x.device)].cpu()
    w_host = w.weight.cpu()
    if w.op == "rms_norm":
        y = ks.rms_norm(x, wt, w.eps)
        torch.cuda.synchronize()
        y_host = y.cpu() if rows_idx is None else y[rows_idx.to(device)].cpu()
        ref, _ = oracle.rms_norm(x_host, w_host, w.eps)
        compare_output(y_host, ref, w.dtype, w.hidden, name)
        return {"y": y, "x": x}
    r = w.residual.to(device, copy=True)
    r_host = w.residual.cpu() if rows_idx is None else w.residual[rows_idx.to(w.residual.device)].cpu()
    ks.fused_add_rms_norm(x, r, wt, w.eps)
    torch.cuda.synchronize()
    xo = x.cpu() if rows_idx is None else x[rows_idx.to(device)].cpu()
    ro = r.cpu() if rows_idx is None else r[rows_idx.to(device)].cpu()
    ref_x, ref_r, _ = oracle.fused_add_rms_norm(x_host, r_host, w_host, w.eps)
    assert bits_equal(ro, ref_r), f"{name}: residual not bit-exact"
    record(name + " residual", bit_exact=True, n=ro.numel())
    compare_output(xo, ref_x, w.dtype, w.hidden, name)
    return {"x": x, "r": r}
