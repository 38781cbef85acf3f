"""ctypes binding of libks's C ABI (include/ks.h), one Python function per C entry point, with
the same names. Argument marshalling only: pointers and sizes in, a status out.

The library is loaded on first use. If it has not been built there is no fallback: the call
raises ``KsLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libks.so")

KS_DTYPE_F32, KS_DTYPE_F16, KS_DTYPE_BF16 = 0, 1, 2
KS_SUCCESS, KS_ERR_INVALID_ARGUMENT, KS_ERR_UNSUPPORTED_DTYPE, KS_ERR_OVERLAP, KS_ERR_CUDA = range(5)
(KS_KERNEL_NONE, KS_KERNEL_WARP_ROW, KS_KERNEL_CTA_ROW, KS_KERNEL_SCALAR, KS_KERNEL_BULK_ROW,
 KS_KERNEL_CLUSTER_ROW, KS_KERNEL_TWOPASS_ROW, KS_KERNEL_FLAT) = range(8)
KERNEL_NAMES = {0: "none", 1: "warp_row", 2: "cta_row", 3: "scalar", 4: "bulk_row",
                5: "cluster_row", 6: "twopass_row", 7: "flat"}
# ks_plan_launch's op codes
OP_RMS_NORM, OP_FUSED_ADD_RMS_NORM, OP_SILU_AND_MUL, OP_SOFTMAX, OP_LAYER_NORM = range(5)
KS_FAULT_WAIT_TIMEOUT = 1
KS_PLAN_NO_PREFETCH = 1
KS_PLAN_PDL = 2
KS_PLAN_AFFINE_SMEM = 4
KS_PLAN_SMEM_ROWS = 8
KS_LAUNCH_PDL = 1

# Every symbol include/ks.h declares (checked by the CPU test of the boundary).
EXPORTED = ("ks_rms_norm", "ks_fused_add_rms_norm", "ks_status_string", "ks_last_error",
            "ks_plan_launch", "ks_rms_norm_planned", "ks_fused_add_rms_norm_planned",
            "ks_device_faults", "ks_rms_norm_host", "ks_fused_add_rms_norm_host",
            "ks_host_chunk_rows", "ks_fused_add_rms_norm_host_noalloc", "ks_set_launch_options",
            "ks_get_launch_options", "ks_silu_and_mul", "ks_softmax", "ks_layer_norm",
            "ks_silu_and_mul_planned", "ks_softmax_planned", "ks_layer_norm_planned",
            "ks_version")


class KsLibraryMissing(RuntimeError):
    pass


class KsError(RuntimeError):
    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}")
        self.status = status
        self.name = name
        self.detail = detail


class ks_plan_t(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("vec_per_thread", ctypes.c_int32),
                ("team", ctypes.c_int32), ("block", ctypes.c_int32), ("grid", ctypes.c_int64),
                ("rows_per_pass", ctypes.c_int64), ("stages", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("cluster", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, "?")
        return d


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libks (once). Raises KsLibraryMissing if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise KsLibraryMissing(
                f"{p} is missing: build it with `python -m row_wise_rmsnorm_ks_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.ks_rms_norm.argtypes = [vp, vp, vp, i64, i64, f32, ctypes.c_int, vp]
        lib.ks_rms_norm.restype = ctypes.c_int
        lib.ks_fused_add_rms_norm.argtypes = [vp, vp, vp, i64, i64, f32, ctypes.c_int, vp]
        lib.ks_fused_add_rms_norm.restype = ctypes.c_int
        lib.ks_status_string.argtypes = [ctypes.c_int]
        lib.ks_status_string.restype = ctypes.c_char_p
        lib.ks_last_error.argtypes = []
        lib.ks_last_error.restype = ctypes.c_char_p
        lib.ks_plan_launch.argtypes = [i32, i64, i64, ctypes.c_int, i32, i32, i32,
                                       ctypes.POINTER(ks_plan_t)]
        lib.ks_plan_launch.restype = ctypes.c_int
        PP = ctypes.POINTER(ks_plan_t)
        lib.ks_rms_norm_planned.argtypes = [vp, vp, vp, i64, i64, f32, ctypes.c_int, PP, vp]
        lib.ks_rms_norm_planned.restype = ctypes.c_int
        lib.ks_fused_add_rms_norm_planned.argtypes = [vp, vp, vp, i64, i64, f32, ctypes.c_int,
                                                      PP, vp]
        lib.ks_fused_add_rms_norm_planned.restype = ctypes.c_int
        lib.ks_device_faults.argtypes = [ctypes.POINTER(i32), i32]
        lib.ks_device_faults.restype = ctypes.c_int
        lib.ks_rms_norm_host.argtypes = [vp, vp, vp, i64, i64, f32, ctypes.c_int, vp, i64, vp]
        lib.ks_rms_norm_host.restype = ctypes.c_int
        lib.ks_fused_add_rms_norm_host.argtypes = [vp, vp, vp, i64, i64, f32, ctypes.c_int, vp,
                                                   i64, vp]
        lib.ks_fused_add_rms_norm_host.restype = ctypes.c_int
        lib.ks_host_chunk_rows.argtypes = [i32, i64, ctypes.c_int, i64]
        lib.ks_host_chunk_rows.restype = i64
        lib.ks_fused_add_rms_norm_host_noalloc.argtypes = [vp, vp, vp, i64, i64, f32,
                                                           ctypes.c_int, vp]
        lib.ks_fused_add_rms_norm_host_noalloc.restype = ctypes.c_int
        lib.ks_set_launch_options.argtypes = [i32]
        lib.ks_set_launch_options.restype = ctypes.c_int
        lib.ks_get_launch_options.argtypes = []
        lib.ks_get_launch_options.restype = i32
        lib.ks_silu_and_mul.argtypes = [vp, vp, i64, i64, ctypes.c_int, vp]
        lib.ks_silu_and_mul.restype = ctypes.c_int
        lib.ks_softmax.argtypes = [vp, vp, i64, i64, ctypes.c_int, vp]
        lib.ks_softmax.restype = ctypes.c_int
        lib.ks_layer_norm.argtypes = [vp, vp, vp, vp, i64, i64, f32, ctypes.c_int, vp]
        lib.ks_layer_norm.restype = ctypes.c_int
        lib.ks_silu_and_mul_planned.argtypes = [vp, vp, i64, i64, ctypes.c_int, PP, vp]
        lib.ks_silu_and_mul_planned.restype = ctypes.c_int
        lib.ks_softmax_planned.argtypes = [vp, vp, i64, i64, ctypes.c_int, PP, vp]
        lib.ks_softmax_planned.restype = ctypes.c_int
        lib.ks_layer_norm_planned.argtypes = [vp, vp, vp, vp, i64, i64, f32, ctypes.c_int, PP, vp]
        lib.ks_layer_norm_planned.restype = ctypes.c_int
        lib.ks_version.argtypes = []
        lib.ks_version.restype = i32
        _lib = lib
        return lib


def ks_rms_norm(out: int, x: int, weight: int, rows: int, hidden: int, eps: float, dtype: int,
                stream: int | None) -> int:
    return load().ks_rms_norm(out, x, weight, rows, hidden, eps, dtype, stream)


def ks_fused_add_rms_norm(x: int, residual: int, weight: int, rows: int, hidden: int,
                          eps: float, dtype: int, stream: int | None) -> int:
    return load().ks_fused_add_rms_norm(x, residual, weight, rows, hidden, eps, dtype, stream)


def ks_status_string(status: int) -> str:
    return load().ks_status_string(status).decode()


def ks_last_error() -> str:
    return load().ks_last_error().decode()


def ks_plan_launch(op: int, rows: int, hidden: int, dtype: int, aligned16: bool, sm_count: int,
                   blocks_per_sm: int) -> tuple[int, ks_plan_t]:
    plan = ks_plan_t()
    st = load().ks_plan_launch(op, rows, hidden, dtype, int(bool(aligned16)), sm_count,
                               blocks_per_sm, ctypes.byref(plan))
    return st, plan


def make_plan(kernel: int, vec_per_thread: int, block: int, stages: int = 0,
              grid: int = 0, flags: int = 0, cluster: int = 0, team: int = 0) -> ks_plan_t:
    """A plan for the *_planned entry points (derived fields are recomputed by the library;
    `team` is read for warp rows: lanes per row, 8, 16 or 32, 0 meaning 32)."""
    p = ks_plan_t()
    p.kernel, p.vec_per_thread, p.block, p.stages, p.grid, p.flags, p.cluster, p.team = (
        kernel, vec_per_thread, block, stages, grid, flags, cluster, team)
    return p


def ks_rms_norm_planned(out: int, x: int, weight: int, rows: int, hidden: int, eps: float,
                        dtype: int, plan: ks_plan_t, stream: int | None) -> int:
    return load().ks_rms_norm_planned(out, x, weight, rows, hidden, eps, dtype,
                                      ctypes.byref(plan), stream)


def ks_fused_add_rms_norm_planned(x: int, residual: int, weight: int, rows: int, hidden: int,
                                  eps: float, dtype: int, plan: ks_plan_t,
                                  stream: int | None) -> int:
    return load().ks_fused_add_rms_norm_planned(x, residual, weight, rows, hidden, eps, dtype,
                                                ctypes.byref(plan), stream)


def ks_device_faults(clear: bool = True) -> tuple[int, int]:
    """(status, flags): the device fault words of the current device, OR-ed."""
    flags = ctypes.c_int32(0)
    st = load().ks_device_faults(ctypes.byref(flags), int(bool(clear)))
    return st, flags.value


def ks_rms_norm_host(out: int, x: int, weight: int, rows: int, hidden: int, eps: float,
                     dtype: int, workspace: int, workspace_bytes: int, stream: int | None) -> int:
    return load().ks_rms_norm_host(out, x, weight, rows, hidden, eps, dtype, workspace,
                                   workspace_bytes, stream)


def ks_fused_add_rms_norm_host(x: int, residual: int, weight: int, rows: int, hidden: int,
                               eps: float, dtype: int, workspace: int, workspace_bytes: int,
                               stream: int | None) -> int:
    return load().ks_fused_add_rms_norm_host(x, residual, weight, rows, hidden, eps, dtype,
                                             workspace, workspace_bytes, stream)


def ks_host_chunk_rows(op: int, hidden: int, dtype: int, workspace_bytes: int) -> int:
    return load().ks_host_chunk_rows(op, hidden, dtype, workspace_bytes)


def ks_fused_add_rms_norm_host_noalloc(x: int, residual: int, weight: int, rows: int, hidden: int,
                                       eps: float, dtype: int, stream: int | None) -> int:
    """The staged host-buffer fused op on the library's built-in 24 MiB device scratch, for
    callers that may not allocate device memory themselves."""
    return load().ks_fused_add_rms_norm_host_noalloc(x, residual, weight, rows, hidden, eps, dtype,
                                                     stream)


def ks_set_launch_options(options: int) -> int:
    return load().ks_set_launch_options(options)


def ks_get_launch_options() -> int:
    return load().ks_get_launch_options()


def ks_silu_and_mul(out: int, x: int, rows: int, d: int, dtype: int, stream: int | None) -> int:
    return load().ks_silu_and_mul(out, x, rows, d, dtype, stream)


def ks_softmax(out: int, x: int, rows: int, hidden: int, dtype: int, stream: int | None) -> int:
    return load().ks_softmax(out, x, rows, hidden, dtype, stream)


def ks_layer_norm(out: int, x: int, weight: int | None, bias: int | None, rows: int, hidden: int,
                  eps: float, dtype: int, stream: int | None) -> int:
    return load().ks_layer_norm(out, x, weight, bias, rows, hidden, eps, dtype, stream)


def ks_silu_and_mul_planned(out: int, x: int, rows: int, d: int, dtype: int, plan: ks_plan_t,
                            stream: int | None) -> int:
    return load().ks_silu_and_mul_planned(out, x, rows, d, dtype, ctypes.byref(plan), stream)


def ks_softmax_planned(out: int, x: int, rows: int, hidden: int, dtype: int, plan: ks_plan_t,
                       stream: int | None) -> int:
    return load().ks_softmax_planned(out, x, rows, hidden, dtype, ctypes.byref(plan), stream)


def ks_layer_norm_planned(out: int, x: int, weight: int | None, bias: int | None, rows: int,
                          hidden: int, eps: float, dtype: int, plan: ks_plan_t,
                          stream: int | None) -> int:
    return load().ks_layer_norm_planned(out, x, weight, bias, rows, hidden, eps, dtype,
                                        ctypes.byref(plan), stream)


def ks_version() -> int:
    return load().ks_version()


def check(status: int) -> None:
    """Raise KsError for a non-success status, with the library's detail string."""
    if status != KS_SUCCESS:
        raise KsError(status, ks_status_string(status), ks_last_error())
