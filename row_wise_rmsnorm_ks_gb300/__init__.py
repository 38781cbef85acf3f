"""Row-wise RMSNorm and fused residual-add RMSNorm for NVIDIA GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind the C ABI of ``libks`` (include/ks.h).
This package is the thin Python binding over it: it marshals torch tensors into pointers and
sizes and never computes anything itself. There is no CPU fallback: without the built library
every op raises ``KsLibraryMissing``.
"""
from ._abi import KsError, KsLibraryMissing  # noqa: F401
from .ops import (fused_add_rms_norm, fused_add_rms_norm_host, layer_norm,  # noqa: F401
                  rms_norm, rms_norm_host, silu_and_mul, softmax)

__all__ = ["rms_norm", "fused_add_rms_norm", "rms_norm_host", "fused_add_rms_norm_host",
           "silu_and_mul", "softmax", "layer_norm", "KsError", "KsLibraryMissing"]
