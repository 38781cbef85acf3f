"""Tensor-level API over the C ABI, with Kernscope's signatures ("API contract"):

    rms_norm(x, weight, eps=1e-6) -> y
    fused_add_rms_norm(x, residual, weight, eps=1e-6) -> None   (x and residual updated in place)

    rms_norm_host(x, weight, eps=1e-6, *, out=None, workspace=None) -> out
    fused_add_rms_norm_host(x, residual, weight, eps=1e-6, *, workspace=None) -> None
(the last two take rows in host memory: without a workspace the kernels read and write pinned
host rows directly over the host link; with a device workspace the library copies them through
it in overlapping chunks).

Checks follow Kernscope "API contract / Inputs": x is (..., hidden) with a non-empty last
dimension, weight is (hidden,), tensors are contiguous CUDA tensors of one dtype (fp16, bf16 or
fp32) on one device, eps is finite and positive, the fused op's residual has x's shape and the
storage of x, residual and weight does not overlap; tensors that require grad are rejected
(inference only). The leading dimensions are flattened into rows. Every launch goes through
libks on the tensor's device and the current torch stream; nothing is computed here.
"""
from __future__ import annotations

import math

import torch

from . import _abi

_DTYPES = {torch.float32: _abi.KS_DTYPE_F32, torch.float16: _abi.KS_DTYPE_F16,
           torch.bfloat16: _abi.KS_DTYPE_BF16}


def _check(x: torch.Tensor, weight: torch.Tensor, eps: float, names=("x", "weight")):
    if not isinstance(x, torch.Tensor) or not isinstance(weight, torch.Tensor):
        raise TypeError("x and weight must be torch tensors")
    if x.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {x.dtype}; use float16, bfloat16 or float32")
    if weight.dtype != x.dtype:
        raise TypeError(f"{names[1]} dtype {weight.dtype} differs from {names[0]} dtype {x.dtype}")
    if x.device.type != "cuda" or weight.device != x.device:
        raise ValueError("tensors must be CUDA tensors on one device (there is no CPU path)")
    if x.dim() < 1 or x.shape[-1] == 0:
        raise ValueError("the last dimension of x must be non-empty")
    if weight.dim() != 1 or weight.shape[0] != x.shape[-1]:
        raise ValueError(f"weight must have shape ({x.shape[-1]},), got {tuple(weight.shape)}")
    if not x.is_contiguous() or not weight.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if torch.is_grad_enabled() and (x.requires_grad or weight.requires_grad):
        raise RuntimeError("these kernels are inference-only: inputs must not require grad")
    if not (isinstance(eps, (int, float)) and math.isfinite(eps) and eps > 0):
        raise ValueError("eps must be finite and positive")


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def rms_norm(x: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6, *,
             out: torch.Tensor | None = None) -> torch.Tensor:
    """y = cast(fp32(x) * rsqrt(mean(fp32(x)^2) + eps) * fp32(weight)) per row. `out` may be x
    itself (in place) or a new contiguous tensor of x's shape and dtype."""
    _check(x, weight, eps)
    if out is None:
        out = torch.empty_like(x)
    elif (out.shape != x.shape or out.dtype != x.dtype or out.device != x.device
          or not out.is_contiguous()):
        raise ValueError("out must be a contiguous tensor with x's shape, dtype and device")
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    with torch.cuda.device(x.device):
        _abi.check(_abi.ks_rms_norm(out.data_ptr(), x.data_ptr(), weight.data_ptr(), rows, hidden,
                                    float(eps), _DTYPES[x.dtype], _stream(x.device)))
    return out


def fused_add_rms_norm(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor,
                       eps: float = 1e-6) -> None:
    """In place: residual <- cast(fp32(x) + fp32(residual)); x <- RMSNorm of the FP32 sum
    times fp32(weight). Returns None."""
    _check(x, weight, eps)
    if not isinstance(residual, torch.Tensor) or residual.shape != x.shape:
        raise ValueError("residual must have the same shape as x")
    if residual.dtype != x.dtype or residual.device != x.device or not residual.is_contiguous():
        raise ValueError("residual must be contiguous, with x's dtype and device")
    if torch.is_grad_enabled() and residual.requires_grad:
        raise RuntimeError("these kernels are inference-only: inputs must not require grad")
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    with torch.cuda.device(x.device):
        _abi.check(_abi.ks_fused_add_rms_norm(x.data_ptr(), residual.data_ptr(),
                                              weight.data_ptr(), rows, hidden, float(eps),
                                              _DTYPES[x.dtype], _stream(x.device)))
    return None


def _check_host(x: torch.Tensor, weight: torch.Tensor, workspace: torch.Tensor, eps: float):
    if not isinstance(x, torch.Tensor) or x.device.type != "cpu":
        raise ValueError("x must be a CPU tensor (pin it for the copies to overlap)")
    if x.dtype not in _DTYPES or weight.dtype != x.dtype:
        raise TypeError("x and weight must share a dtype: float16, bfloat16 or float32")
    if weight.device.type != "cuda" or weight.dim() != 1 or weight.shape[0] != x.shape[-1]:
        raise ValueError("weight must be a CUDA tensor of shape (hidden,)")
    if workspace is not None and (not isinstance(workspace, torch.Tensor)
                                  or workspace.device != weight.device
                                  or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on weight's device")
    if workspace is None and not x.is_pinned():
        raise ValueError("without a workspace the host rows must be pinned")
    if not (x.is_contiguous() and weight.is_contiguous()):
        raise ValueError("tensors must be contiguous")
    if x.dim() < 1 or x.shape[-1] == 0:
        raise ValueError("the last dimension of x must be non-empty")
    if not (isinstance(eps, (int, float)) and math.isfinite(eps) and eps > 0):
        raise ValueError("eps must be finite and positive")


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def rms_norm_host(x: torch.Tensor, weight: torch.Tensor, eps: float = 1e-6, *,
                  workspace: torch.Tensor | None = None,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """RMSNorm of host rows through the device: returns `out` (a host tensor, x's shape; may be
    x). Ordered on the current stream of weight's device; synchronise it before reading `out`."""
    _check_host(x, weight, workspace, eps)
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, pin_memory=x.is_pinned())
    elif out.shape != x.shape or out.dtype != x.dtype or out.device.type != "cpu":
        raise ValueError("out must be a CPU tensor with x's shape and dtype")
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    with torch.cuda.device(weight.device):
        _abi.check(_abi.ks_rms_norm_host(out.data_ptr(), x.data_ptr(), weight.data_ptr(), rows,
                                         hidden, float(eps), _DTYPES[x.dtype], *_ws(workspace),
                                         _stream(weight.device)))
    return out


def fused_add_rms_norm_host(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor,
                            eps: float = 1e-6, *, workspace: torch.Tensor | None = None) -> None:
    """Fused residual-add RMSNorm of host rows through the device, in place on both host
    tensors. Ordered on the current stream of weight's device; synchronise before reading."""
    _check_host(x, weight, workspace, eps)
    if (not isinstance(residual, torch.Tensor) or residual.shape != x.shape
            or residual.dtype != x.dtype or residual.device.type != "cpu"
            or not residual.is_contiguous()):
        raise ValueError("residual must be a contiguous CPU tensor with x's shape and dtype")
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    with torch.cuda.device(weight.device):
        _abi.check(_abi.ks_fused_add_rms_norm_host(x.data_ptr(), residual.data_ptr(),
                                                   weight.data_ptr(), rows, hidden, float(eps),
                                                   _DTYPES[x.dtype], *_ws(workspace),
                                                   _stream(weight.device)))
    return None


# ------------------------------------------------------------------ the next operators

def _check_plain(x: torch.Tensor, name="x"):
    if not isinstance(x, torch.Tensor) or x.dtype not in _DTYPES:
        raise TypeError(f"{name} must be a float16, bfloat16 or float32 tensor")
    if x.device.type != "cuda":
        raise ValueError("tensors must be CUDA tensors (there is no CPU path)")
    if not x.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if x.dim() < 1 or x.shape[-1] == 0:
        raise ValueError("the last dimension must be non-empty")
    if torch.is_grad_enabled() and x.requires_grad:
        raise RuntimeError("these kernels are inference-only: inputs must not require grad")


def silu_and_mul(x: torch.Tensor) -> torch.Tensor:
    """SwiGLU (Kernscope, "Numerical contract / SwiGLU activation"): x of shape (..., 2D) gives
    cast(gate * sigmoid(gate) * up) of shape (..., D), gate = x[..., :D], up = x[..., D:], FP32
    throughout. x is read-only; D may be odd; leading dimensions may be empty."""
    _check_plain(x)
    if x.shape[-1] % 2:
        raise ValueError("the last dimension of x must be even")
    d = x.shape[-1] // 2
    out = torch.empty(tuple(x.shape[:-1]) + (d,), dtype=x.dtype, device=x.device)
    rows = x.numel() // x.shape[-1]
    with torch.cuda.device(x.device):
        _abi.check(_abi.ks_silu_and_mul(out.data_ptr(), x.data_ptr(), rows, d, _DTYPES[x.dtype],
                                        _stream(x.device)))
    return out


def softmax(x: torch.Tensor, *, out: torch.Tensor | None = None) -> torch.Tensor:
    """Softmax over the last dimension (Kernscope, "Numerical contract / Softmax"), FP32
    max/exp/sum/divide, cast back; rows with NaN or +inf, or all -inf, come out NaN."""
    _check_plain(x)
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or out.device != x.device:
        raise ValueError("out must match x in shape, dtype and device")
    hidden = x.shape[-1]
    with torch.cuda.device(x.device):
        _abi.check(_abi.ks_softmax(out.data_ptr(), x.data_ptr(), x.numel() // hidden, hidden,
                                   _DTYPES[x.dtype], _stream(x.device)))
    return out


def layer_norm(x: torch.Tensor, weight: torch.Tensor | None = None,
               bias: torch.Tensor | None = None, eps: float = 1e-5, *,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """LayerNorm over the last dimension with FP32 steps:
    cast((((x - mean) * rsqrt(var + eps)) * weight) + bias); weight and bias optional."""
    _check_plain(x)
    hidden = x.shape[-1]
    for t, n in ((weight, "weight"), (bias, "bias")):
        if t is not None and (t.dtype != x.dtype or t.device != x.device or t.dim() != 1
                              or t.shape[0] != hidden or not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous ({hidden},) tensor of x's dtype and device")
    if not (isinstance(eps, (int, float)) and math.isfinite(eps) and eps > 0):
        raise ValueError("eps must be finite and positive")
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        _abi.check(_abi.ks_layer_norm(out.data_ptr(), x.data_ptr(),
                                      weight.data_ptr() if weight is not None else None,
                                      bias.data_ptr() if bias is not None else None,
                                      x.numel() // hidden, hidden, float(eps), _DTYPES[x.dtype],
                                      _stream(x.device)))
    return out
