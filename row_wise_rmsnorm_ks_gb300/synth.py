"""Seeded synthetic inputs for the RMSNorm workloads.

This module only draws random numbers and casts them to the input dtype. It holds none of the
method's arithmetic, so both the CUDA path's tests and the oracle can take their inputs from it.

Workload shapes and laws (the pages' own shapes: Kernscope "CUDA performance" 512x1024; Triton
Kernel Lab "Measured Result" 128x1024, 512x4096, 2048x4096 and "Decode Kernel Results" 4x1536;
Triton Kernels "Benchmark results" hidden 4096 x seq 2048), widened to the sizes a GB300 holds:

  small         rms_norm bf16 [128, 1024], x ~ N(0,1), weight = 1 + 0.1 N(0,1), eps 1e-6
  medium        rms_norm fp16/bf16 [2048, 4096], x ~ N(0,1) with one constant row and one zero
                row at seeded positions, eps 1e-6
  fused         fused_add_rms_norm bf16 [512, 4096], x ~ N(0,1), residual ~ N(0, variance 4);
                decode shape [4, 1536] with the same laws, eps 1e-6
  prefill       both ops bf16 [rows, 8192] (rows up to 32768), x, residual ~ N(0,1), eps 1e-5
  wide          both ops fp16/bf16, hidden in {1536, 5120, 7168, 14336, 16384} x rows in
                {1, 7, 333, 65536}; x and residual ~ Student-t(3), with max(1, round(rows/100))
                seeded rows scaled by 1e3; fp16 inputs saturated to +-65504 before the cast
                (so no input is inf); eps 1e-6

Seeds: x 1234, residual 1235, weight 1236, row positions 1237. Host generation uses numpy's
PCG64 ``default_rng``; Student-t(3) is Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3) from four independent
standard normals. ``device=`` generation draws the same laws with torch's generator on a CUDA
device (used only where a host draw of gigabytes would dominate a test's run time).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

SEED_X = 1234
SEED_RESIDUAL = 1235
SEED_WEIGHT = 1236
SEED_ROWS = 1237

FP16_MAX = 65504.0

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def dtype_of(name_or_dtype) -> torch.dtype:
    if isinstance(name_or_dtype, torch.dtype):
        return name_or_dtype
    return DTYPES[name_or_dtype]


def cast(a32: np.ndarray | torch.Tensor, dtype) -> torch.Tensor:
    """fp32 draws -> input dtype (round to nearest even, torch's cast). fp16 draws are first
    saturated to +-65504 so the heavy-tailed laws put no inf into fp16 inputs."""
    dtype = dtype_of(dtype)
    t = torch.from_numpy(np.ascontiguousarray(a32)) if isinstance(a32, np.ndarray) else a32
    t = t.to(torch.float32)
    if dtype == torch.float16:
        t = t.clamp(-FP16_MAX, FP16_MAX)
    return t.to(dtype)


# ------------------------------------------------------------------------------------ host laws

def normal_np(shape, seed: int, std: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(int(np.prod(shape)), dtype=np.float32).reshape(shape)
    if std != 1.0:
        a *= np.float32(std)
    return a


def student_t3_np(shape, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    n = int(np.prod(shape))
    z = rng.standard_normal(n, dtype=np.float32)
    c = np.zeros(n, dtype=np.float32)
    for _ in range(3):
        g = rng.standard_normal(n, dtype=np.float32)
        c += g * g
    return (z / np.sqrt(c / np.float32(3.0))).reshape(shape)


def outlier_rows(rows: int, seed: int = SEED_ROWS, frac: float = 0.01) -> np.ndarray:
    """Seeded positions of the rows scaled by 1e3 in the wide sweep."""
    if rows == 0:
        return np.zeros(0, dtype=np.int64)
    k = max(1, int(round(frac * rows)))
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(rows, size=k, replace=False)).astype(np.int64)


def special_rows(rows: int, seed: int = SEED_ROWS):
    """Seeded positions (const_row, zero_row) and the constant c ~ N(0,1) for the medium case."""
    rng = np.random.default_rng(seed)
    pos = rng.choice(rows, size=2, replace=False)
    c = np.float32(rng.standard_normal())
    return int(pos[0]), int(pos[1]), c


def weight(hidden: int, dtype, seed: int = SEED_WEIGHT) -> torch.Tensor:
    """weight = 1 + 0.1 N(0,1), cast to dtype."""
    w = np.float32(1.0) + np.float32(0.1) * normal_np((hidden,), seed)
    return cast(w, dtype)


# ------------------------------------------------------------------------------ workload object

@dataclass
class Workload:
    name: str
    op: str                      # "rms_norm" or "fused_add_rms_norm"
    dtype: torch.dtype
    x: torch.Tensor              # [rows, hidden] CPU (or device when generated there)
    weight: torch.Tensor         # [hidden]
    eps: float
    residual: torch.Tensor | None = None
    notes: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.x.shape[0]

    @property
    def hidden(self) -> int:
        return self.x.shape[-1]


def small() -> Workload:
    return Workload("small rms_norm bf16 [128,1024]", "rms_norm", torch.bfloat16,
                    cast(normal_np((128, 1024), SEED_X), torch.bfloat16),
                    weight(1024, torch.bfloat16), 1e-6)


def medium(dtype="bf16", rows: int = 2048, hidden: int = 4096) -> Workload:
    dtype = dtype_of(dtype)
    x = normal_np((rows, hidden), SEED_X)
    ci, zi, c = special_rows(rows)
    x[ci, :] = c
    x[zi, :] = 0.0
    xt = cast(x, dtype)
    return Workload(f"medium rms_norm {dtype} [{rows},{hidden}]", "rms_norm", dtype, xt,
                    weight(hidden, dtype), 1e-6,
                    notes={"const_row": ci, "zero_row": zi, "c": float(xt[ci, 0].float())})


def fused(rows: int = 512, hidden: int = 4096, dtype="bf16") -> Workload:
    dtype = dtype_of(dtype)
    return Workload(f"fused_add_rms_norm {dtype} [{rows},{hidden}]", "fused_add_rms_norm", dtype,
                    cast(normal_np((rows, hidden), SEED_X), dtype), weight(hidden, dtype), 1e-6,
                    residual=cast(normal_np((rows, hidden), SEED_RESIDUAL, std=2.0), dtype))


def decode() -> Workload:
    w = fused(4, 1536)
    w.name = "decode fused_add_rms_norm bf16 [4,1536]"
    return w


def prefill(op: str, rows: int = 32768, hidden: int = 8192, dtype="bf16") -> Workload:
    dtype = dtype_of(dtype)
    x = cast(normal_np((rows, hidden), SEED_X), dtype)
    r = cast(normal_np((rows, hidden), SEED_RESIDUAL), dtype) if op != "rms_norm" else None
    return Workload(f"prefill {op} {dtype} [{rows},{hidden}]", op, dtype, x,
                    weight(hidden, dtype), 1e-5, residual=r)


def _scale_rows(a: np.ndarray, rows_idx: np.ndarray) -> np.ndarray:
    a[rows_idx, :] *= np.float32(1e3)
    return a


def wide(op: str, hidden: int, rows: int, dtype="bf16") -> Workload:
    dtype = dtype_of(dtype)
    idx = outlier_rows(rows)
    x = cast(_scale_rows(student_t3_np((rows, hidden), SEED_X), idx), dtype)
    r = None
    if op != "rms_norm":
        r = cast(_scale_rows(student_t3_np((rows, hidden), SEED_RESIDUAL), idx), dtype)
    return Workload(f"wide {op} {dtype} [{rows},{hidden}]", op, dtype, x, weight(hidden, dtype),
                    1e-6, residual=r, notes={"outlier_rows": idx.tolist()})


# --------------------------------------------------------------------------- device generation

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_dev(shape, seed: int, device, std: float = 1.0) -> torch.Tensor:
    t = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return t.mul_(std) if std != 1.0 else t


def student_t3_dev(shape, seed: int, device) -> torch.Tensor:
    g = _gen(device, seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    c = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(3):
        n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        c.addcmul_(n, n)
    return z.div_(c.div_(3.0).sqrt_())


def wide_device(op: str, hidden: int, rows: int, dtype, device) -> Workload:
    """The wide-sweep laws drawn on `device` (for the multi-gigabyte cases)."""
    dtype = dtype_of(dtype)
    idx = outlier_rows(rows)
    it = torch.from_numpy(idx).to(device)

    def draw(seed):
        a = student_t3_dev((rows, hidden), seed, device)
        a[it] = a[it] * 1e3
        return cast(a, dtype)

    x = draw(SEED_X)
    r = draw(SEED_RESIDUAL) if op != "rms_norm" else None
    return Workload(f"wide {op} {dtype} [{rows},{hidden}] (device draw)", op, dtype, x,
                    weight(hidden, dtype).to(device), 1e-6, residual=r,
                    notes={"outlier_rows": idx.tolist()})


def prefill_device(op: str, rows: int, hidden: int, dtype, device) -> Workload:
    dtype = dtype_of(dtype)
    x = cast(normal_dev((rows, hidden), SEED_X, device), dtype)
    r = cast(normal_dev((rows, hidden), SEED_RESIDUAL, device), dtype) if op != "rms_norm" else None
    return Workload(f"prefill {op} {dtype} [{rows},{hidden}] (device draw)", op, dtype, x,
                    weight(hidden, dtype).to(device), 1e-5, residual=r)
