"""CPU oracle for row-wise RMSNorm and the fused residual-add RMSNorm.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package. The product path (the CUDA library and its binding)
never calls it, and it imports nothing from the product: the two share no code. Inputs come
from the seeded generators in ``row_wise_rmsnorm_ks_gb300.synth``, which hold none of the
method's arithmetic.

The arithmetic lives in ``ks_oracle.c`` (plain C, single-threaded, built with no FMA
contraction). This module only marshals CPU torch tensors into it. Each function follows
Kernscope, "Numerical contract" (RMSNorm; Fused residual-add RMSNorm; SwiGLU activation;
Softmax) or, for LayerNorm (only named on kernel-set's operator list), the standard definition
with the same FP32 discipline; the readings taken where a contract is silent are listed at the
top of ``ks_oracle.c`` and beside each function.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests
(tests/test_oracle_*.py) against exact rationals, closed forms, invariants, a float64 brute
force and torch's own casts; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes

import torch

from . import build as _build

_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        i64, p, f32, f64, c_int = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_int)
        lib.oracle_rms_norm.argtypes = [p, p, p, p, i64, i64, f32, c_int]
        lib.oracle_rms_norm.restype = None
        lib.oracle_fused_add_rms_norm.argtypes = [p, p, p, p, i64, i64, f32, c_int]
        lib.oracle_fused_add_rms_norm.restype = c_int
        lib.oracle_rms_norm_f64.argtypes = [p, p, p, i64, i64, f64, c_int]
        lib.oracle_rms_norm_f64.restype = None
        lib.oracle_fused_add_rms_norm_f64.argtypes = [p, p, p, p, p, i64, i64, f64, c_int]
        lib.oracle_fused_add_rms_norm_f64.restype = None
        lib.oracle_decode.argtypes = [p, p, i64, c_int]
        lib.oracle_decode.restype = None
        lib.oracle_encode.argtypes = [p, p, i64, c_int]
        lib.oracle_encode.restype = None
        lib.oracle_rsqrt.argtypes = [p, p, i64]
        lib.oracle_rsqrt.restype = None
        lib.oracle_silu_and_mul.argtypes = [p, p, p, i64, i64, c_int]
        lib.oracle_silu_and_mul.restype = None
        lib.oracle_softmax.argtypes = [p, p, p, i64, i64, c_int]
        lib.oracle_softmax.restype = None
        lib.oracle_layer_norm.argtypes = [p, p, p, p, p, i64, i64, f32, c_int]
        lib.oracle_layer_norm.restype = None
        lib.oracle_version.restype = c_int
        _lib = lib
    return _lib


def _check_rows(x: torch.Tensor, weight: torch.Tensor):
    if x.device.type != "cpu" or weight.device.type != "cpu":
        raise ValueError("the oracle runs on CPU tensors only")
    if x.dtype not in _CODES or weight.dtype != x.dtype:
        raise ValueError(f"unsupported dtype pair {x.dtype}/{weight.dtype}")
    H = weight.numel()
    if x.shape[-1] != H:
        raise ValueError("last dim of x must equal weight.numel()")
    return x.reshape(-1, H).contiguous(), weight.contiguous(), H


def rms_norm(x: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6):
    """RMSNorm per the contract. Returns (y, u): y in x's dtype and shape, u the fp32 values
    before the final cast. Inputs are not modified."""
    lib = _load()
    x2, w, H = _check_rows(x, weight)
    y = torch.empty_like(x2)
    u = torch.empty(x2.shape, dtype=torch.float32)
    lib.oracle_rms_norm(x2.data_ptr(), w.data_ptr(), y.data_ptr(), u.data_ptr(),
                        x2.shape[0], H, float(eps), _CODES[x.dtype])
    return y.reshape(x.shape), u.reshape(x.shape)


def fused_add_rms_norm(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor,
                       eps: float = 1e-6):
    """Fused residual-add RMSNorm per the contract. Works on copies and returns
    (x_out, residual_out, u), u being the fp32 normalised values before the final cast."""
    lib = _load()
    x2, w, H = _check_rows(x, weight)
    if residual.shape != x.shape or residual.dtype != x.dtype:
        raise ValueError("residual must match x in shape and dtype")
    xo = x2.clone()
    ro = residual.reshape(-1, H).contiguous().clone()
    u = torch.empty(x2.shape, dtype=torch.float32)
    rc = lib.oracle_fused_add_rms_norm(xo.data_ptr(), ro.data_ptr(), w.data_ptr(), u.data_ptr(),
                                       x2.shape[0], H, float(eps), _CODES[x.dtype])
    if rc != 0:
        raise MemoryError("oracle could not allocate its row buffer")
    return xo.reshape(x.shape), ro.reshape(x.shape), u.reshape(x.shape)


def rms_norm_f64(x: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    """The float64 twin of rms_norm: unrounded double results. eps is taken at its fp32 value,
    as the contract adds it in fp32."""
    lib = _load()
    x2, w, H = _check_rows(x, weight)
    yd = torch.empty(x2.shape, dtype=torch.float64)
    eps32 = float(torch.tensor(eps, dtype=torch.float32))
    lib.oracle_rms_norm_f64(x2.data_ptr(), w.data_ptr(), yd.data_ptr(), x2.shape[0], H, eps32,
                            _CODES[x.dtype])
    return yd.reshape(x.shape)


def fused_add_rms_norm_f64(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor,
                           eps: float = 1e-6):
    """The float64 twin of fused_add_rms_norm: returns (y_double, s_double)."""
    lib = _load()
    x2, w, H = _check_rows(x, weight)
    r2 = residual.reshape(-1, H).contiguous()
    yd = torch.empty(x2.shape, dtype=torch.float64)
    sd = torch.empty(x2.shape, dtype=torch.float64)
    eps32 = float(torch.tensor(eps, dtype=torch.float32))
    lib.oracle_fused_add_rms_norm_f64(x2.data_ptr(), r2.data_ptr(), w.data_ptr(), yd.data_ptr(),
                                      sd.data_ptr(), x2.shape[0], H, eps32, _CODES[x.dtype])
    return yd.reshape(x.shape), sd.reshape(x.shape)


def silu_and_mul(x: torch.Tensor):
    """SwiGLU per Kernscope's contract on x of shape (..., 2d). Returns (out, u): out of shape
    (..., d) in x's dtype, u the fp32 values before the cast."""
    lib = _load()
    if x.device.type != "cpu" or x.dtype not in _CODES or x.shape[-1] % 2:
        raise ValueError("x must be a CPU fp16/bf16/fp32 tensor with an even last dimension")
    d = x.shape[-1] // 2
    x2 = x.reshape(-1, 2 * d).contiguous()
    out = torch.empty((x2.shape[0], d), dtype=x.dtype)
    u = torch.empty((x2.shape[0], d), dtype=torch.float32)
    lib.oracle_silu_and_mul(x2.data_ptr(), out.data_ptr(), u.data_ptr(), x2.shape[0], d,
                            _CODES[x.dtype])
    shape = tuple(x.shape[:-1]) + (d,)
    return out.reshape(shape), u.reshape(shape)


def softmax(x: torch.Tensor):
    """Softmax over the last axis per Kernscope's contract. Returns (out, u)."""
    lib = _load()
    if x.device.type != "cpu" or x.dtype not in _CODES or x.shape[-1] == 0:
        raise ValueError("x must be a CPU fp16/bf16/fp32 tensor with a non-empty last dimension")
    H = x.shape[-1]
    x2 = x.reshape(-1, H).contiguous()
    out = torch.empty_like(x2)
    u = torch.empty(x2.shape, dtype=torch.float32)
    lib.oracle_softmax(x2.data_ptr(), out.data_ptr(), u.data_ptr(), x2.shape[0], H,
                       _CODES[x.dtype])
    return out.reshape(x.shape), u.reshape(x.shape)


def layer_norm(x: torch.Tensor, weight: torch.Tensor | None, bias: torch.Tensor | None,
               eps: float = 1e-5):
    """LayerNorm over the last axis (the standard definition, FP32 steps). Returns (out, u)."""
    lib = _load()
    H = x.shape[-1]
    for t in (weight, bias):
        if t is not None and (t.dtype != x.dtype or t.numel() != H or t.device.type != "cpu"):
            raise ValueError("weight and bias must be CPU tensors of x's dtype and shape (H,)")
    x2 = x.reshape(-1, H).contiguous()
    out = torch.empty_like(x2)
    u = torch.empty(x2.shape, dtype=torch.float32)
    keep = (weight.contiguous() if weight is not None else None,
            bias.contiguous() if bias is not None else None)
    wp = keep[0].data_ptr() if keep[0] is not None else None
    bp = keep[1].data_ptr() if keep[1] is not None else None
    lib.oracle_layer_norm(x2.data_ptr(), wp, bp, out.data_ptr(), u.data_ptr(), x2.shape[0], H,
                          float(eps), _CODES[x.dtype])
    return out.reshape(x.shape), u.reshape(x.shape)


def decode(t: torch.Tensor) -> torch.Tensor:
    """Exact float64 values of a bf16/fp16/fp32 tensor, by the oracle's own bit decoding."""
    lib = _load()
    t = t.contiguous()
    out = torch.empty(t.shape, dtype=torch.float64)
    lib.oracle_decode(t.data_ptr(), out.data_ptr(), t.numel(), _CODES[t.dtype])
    return out


def encode(v: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Round float64 values to `dtype`, nearest-even, by the oracle's own rounding."""
    lib = _load()
    v = v.to(torch.float64).contiguous()
    out = torch.empty(v.shape, dtype=dtype)
    lib.oracle_encode(v.data_ptr(), out.data_ptr(), v.numel(), _CODES[dtype])
    return out


def rsqrt(v: torch.Tensor) -> torch.Tensor:
    """Correctly rounded fp32 1/sqrt(v) for an fp32 tensor."""
    lib = _load()
    v = v.to(torch.float32).contiguous()
    out = torch.empty_like(v)
    lib.oracle_rsqrt(v.data_ptr(), out.data_ptr(), v.numel())
    return out


def version() -> int:
    return _load().oracle_version()
