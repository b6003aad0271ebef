"""Python binding of the GB300 fused gated-activation library.

Argument marshalling only: every step of the activations runs in the CUDA
library ``_lib/libgated_act.so`` (built from ``csrc/`` by ``build.py``) behind
the C ABI declared in ``include/gated_act.h``.  PyTorch supplies memory
(device, or page-locked host memory the kernels read and write in place) and
the current stream.  There is no CPU or eager fallback: if the library is
missing or a call fails, this module raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

LIB_PATH = _build.LIB

OK = 0
ERR_NULL, ERR_SIZE, ERR_STRIDE, ERR_TOO_LARGE = -1, -2, -3, -4
ERR_OVERLAP, ERR_VARIANT, ERR_CUDA, ERR_ALIGN, ERR_DTYPE, ERR_HOST = -5, -6, -7, -8, -9, -10
ERR_SCRATCH, ERR_DEVICE = -11, -12

BF16, F16, F32 = 0, 1, 2
_DTYPE_CODE = {torch.bfloat16: BF16, torch.float16: F16, torch.float32: F32}

VARIANT_AUTO, VARIANT_WARP_ROWS, VARIANT_CTA_ROW, VARIANT_SCALAR, VARIANT_TMA_ROWS = 0, 1, 2, 3, 4
VARIANT_PIPE_ROWS, VARIANT_SPLIT_ROWS = 5, 6
VARIANT_NAMES = {0: "auto", 1: "warp_rows", 2: "cta_row", 3: "scalar", 4: "tma_rows", 5: "pipe_rows",
                 6: "split_rows"}

EXPORTED = (
    "gelu_and_mul_sparse", "gelu_and_mul_sparse_typed", "gelu_and_mul_sparse_native",
    "silu_and_mul", "gated_act_status_string",
    "gated_act_last_cuda_error", "gelu_and_mul_sparse_plan", "gelu_and_mul_sparse_plan_ex",
    "gelu_and_mul_sparse_ex",
    "gated_act_device_status", "gated_act_noop", "gated_act_selftest_wait_timeout",
    "silu_and_mul_bounded", "gelu_and_mul",
    "squared_relu", "gelu_and_mul_sparse_workspace_bytes", "gelu_and_mul_sparse_ws",
    "gelu_and_mul_sparse_ws_static", "gated_act_selftest_wait_timeout_ws",
    "gated_act_selftest_wait_timeout_ex", "gelu_and_mul_sparse_native_plan",
)


class GatedActError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status}: {msg}")
        self.status = status


class Plan(ctypes.Structure):
    """Mirror of ``gated_act_plan``."""

    _fields_ = [("variant", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("vec_per_thread", ctypes.c_int32),
                ("rows_per_cta", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("dynamic_rows", ctypes.c_int32),
                ("grid", ctypes.c_int64), ("smem_bytes", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {"variant": VARIANT_NAMES.get(self.variant, str(self.variant)),
                "cluster": self.cluster, "threads": self.threads,
                "vec_per_thread": self.vec_per_thread, "rows_per_cta": self.rows_per_cta,
                "stages": self.stages, "ctas_per_sm": self.ctas_per_sm,
                "dynamic_rows": self.dynamic_rows, "grid": self.grid,
                "smem_bytes": self.smem_bytes}


_lib: ctypes.CDLL | None = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (once) and declare the C signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"CUDA library {p} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (no fallback exists)")
    lib = ctypes.CDLL(p)
    i64, vp, cvp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.gelu_and_mul_sparse.argtypes = [vp, cvp, i64, i64, i64, ctypes.c_double, vp]
    lib.gelu_and_mul_sparse.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_ex.argtypes = [vp, cvp, i64, i64, i64, ctypes.c_double,
                                           ctypes.c_int, ctypes.c_int, vp]
    lib.gelu_and_mul_sparse_ex.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_plan.argtypes = [cvp, cvp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.POINTER(Plan)]
    lib.gelu_and_mul_sparse_plan_ex.argtypes = [cvp, cvp, i64, i64, i64, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.POINTER(Plan)]
    lib.gelu_and_mul_sparse_plan_ex.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_native_plan.argtypes = [cvp, cvp, i64, i64, i64, ctypes.c_int,
                                                    ctypes.c_int, ctypes.POINTER(Plan)]
    lib.gelu_and_mul_sparse_native_plan.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_typed.argtypes = [vp, cvp, i64, i64, i64, ctypes.c_double,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
    lib.gelu_and_mul_sparse_typed.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_native.argtypes = [vp, cvp, i64, i64, i64, ctypes.c_double,
                                               ctypes.c_int, vp]
    lib.gelu_and_mul_sparse_native.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_plan.restype = ctypes.c_int
    lib.silu_and_mul.argtypes = [vp, cvp, i64, i64, vp]
    lib.silu_and_mul.restype = ctypes.c_int
    lib.gated_act_status_string.argtypes = [ctypes.c_int]
    lib.gated_act_status_string.restype = ctypes.c_char_p
    lib.gated_act_last_cuda_error.argtypes = []
    lib.gated_act_last_cuda_error.restype = ctypes.c_int
    lib.gated_act_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.gated_act_device_status.restype = ctypes.c_int
    lib.gated_act_noop.argtypes = [vp]
    lib.gated_act_noop.restype = ctypes.c_int
    lib.gated_act_selftest_wait_timeout.argtypes = [vp, cvp, i64, i64, ctypes.c_ulonglong, vp]
    lib.gated_act_selftest_wait_timeout.restype = ctypes.c_int
    lib.gated_act_selftest_wait_timeout_ws.argtypes = [vp, cvp, i64, i64, ctypes.c_ulonglong,
                                                       vp, vp]
    lib.gated_act_selftest_wait_timeout_ws.restype = ctypes.c_int
    lib.gated_act_selftest_wait_timeout_ex.argtypes = [vp, cvp, i64, i64, ctypes.c_ulonglong,
                                                       ctypes.c_int, vp, vp]
    lib.gated_act_selftest_wait_timeout_ex.restype = ctypes.c_int
    lib.silu_and_mul_bounded.argtypes = [vp, cvp, i64, i64, cvp, vp]
    lib.silu_and_mul_bounded.restype = ctypes.c_int
    lib.gelu_and_mul.argtypes = [vp, cvp, i64, i64, i64, vp]
    lib.gelu_and_mul.restype = ctypes.c_int
    lib.squared_relu.argtypes = [vp, cvp, i64, i64, vp]
    lib.squared_relu.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_workspace_bytes.argtypes = []
    lib.gelu_and_mul_sparse_workspace_bytes.restype = ctypes.c_size_t
    lib.gelu_and_mul_sparse_ws.argtypes = [vp, cvp, i64, i64, i64, ctypes.c_double, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, vp, vp]
    lib.gelu_and_mul_sparse_ws.restype = ctypes.c_int
    lib.gelu_and_mul_sparse_ws_static.argtypes = [vp, cvp, i64, i64, i64, ctypes.c_double,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
    lib.gelu_and_mul_sparse_ws_static.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().gated_act_status_string(int(status)).decode()


def _check(fn: str, rc: int) -> None:
    if rc != OK:
        msg = status_string(rc)
        if rc == ERR_CUDA:
            msg += f" (cudaError {load_library().gated_act_last_cuda_error()})"
        raise GatedActError(fn, rc, msg)


def _empty_like_rows(x: torch.Tensor, T: int, d: int) -> torch.Tensor:
    """An output [T, d] of x's type where x lives: device, or page-locked host."""
    if x.is_cuda:
        return torch.empty((T, d), dtype=x.dtype, device=x.device)
    return torch.empty((T, d), dtype=x.dtype, pin_memory=True)


def _is_device_or_pinned(x: torch.Tensor) -> bool:
    return x.is_cuda or x.is_pinned()


def _stream_handle(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _rows_view(x: torch.Tensor, dtypes=(torch.bfloat16,)) -> tuple[int, int]:
    """(T, row_stride) for a 2-D device or page-locked tensor whose rows may be strided."""
    if x.dim() != 2:
        raise ValueError("input must be 2-D [T, row_stride]")
    if x.dtype not in dtypes:
        raise TypeError(f"input must be one of {dtypes}")
    if not (x.is_cuda or x.is_pinned()):
        raise ValueError("input must be a CUDA tensor or page-locked host memory "
                         "(the library has no CPU path)")
    if x.stride(1) != 1:
        raise ValueError("input columns must be contiguous")
    return int(x.shape[0]), int(x.stride(0)) if x.shape[0] > 1 else int(x.shape[1])


def workspace_bytes() -> int:
    """Bytes of the workspace ``gelu_and_mul_sparse(..., workspace=)`` takes."""
    return int(load_library().gelu_and_mul_sparse_workspace_bytes())


def new_workspace(device=None) -> torch.Tensor:
    """A zeroed workspace on ``device``.  Calls that share it must run one after
    another on the GPU (one stream, or ordered streams); every completed call
    leaves it zeroed."""
    return torch.zeros(workspace_bytes(), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def gelu_and_mul_sparse(x: torch.Tensor, z: float, d: int | None = None,
                        out: torch.Tensor | None = None, variant: int = VARIANT_AUTO,
                        cluster: int = 0, stream: torch.cuda.Stream | None = None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Sparse GELU gate of ``x`` ([T, >=2d] bf16, fp16 or fp32, on the device or
    in page-locked host memory): returns ``out`` [T, d] of the same type.

    ``d`` defaults to half the row length.  Rows may be strided (x[:, :2d] of a
    wider buffer).  ``variant``/``cluster`` force a launch geometry.
    ``workspace`` (from :func:`new_workspace`) lets the persistent bulk-copy
    geometry hand rows out dynamically; calls sharing one must not overlap.
    """
    T, rs = _rows_view(x, tuple(_DTYPE_CODE))
    if d is None:
        if x.shape[1] % 2:
            raise ValueError("odd row length: pass d explicitly")
        d = int(x.shape[1]) // 2
    if x.shape[1] < 2 * d:
        raise ValueError("rows are shorter than 2d")
    if out is None:
        out = _empty_like_rows(x, T, d)
    elif out.shape != (T, d) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous [T, d] {x.dtype} tensor")
    lib = load_library()
    if workspace is None:
        rc = lib.gelu_and_mul_sparse_typed(out.data_ptr(), x.data_ptr(), T, d, rs, float(z),
                                           _DTYPE_CODE[x.dtype], int(variant), int(cluster),
                                           _stream_handle(stream))
        _check("gelu_and_mul_sparse", rc)
        return out
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < workspace_bytes():
        raise ValueError("workspace must be a device tensor of at least workspace_bytes() bytes")
    rc = lib.gelu_and_mul_sparse_ws(out.data_ptr(), x.data_ptr(), T, d, rs, float(z),
                                    _DTYPE_CODE[x.dtype], int(variant), int(cluster),
                                    workspace.data_ptr(), _stream_handle(stream))
    _check("gelu_and_mul_sparse_ws", rc)
    return out


def gelu_and_mul_sparse_native(x: torch.Tensor, z: float, d: int | None = None,
                               out: torch.Tensor | None = None,
                               stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Native-rounding sparse GELU of ``x`` ([T, >=2d] bf16 or fp16): every
    intermediate rounded to the element type, as separate PyTorch ops round."""
    T, rs = _rows_view(x, (torch.bfloat16, torch.float16))
    if d is None:
        if x.shape[1] % 2:
            raise ValueError("odd row length: pass d explicitly")
        d = int(x.shape[1]) // 2
    if x.shape[1] < 2 * d:
        raise ValueError("rows are shorter than 2d")
    if out is None:
        out = _empty_like_rows(x, T, d)
    elif out.shape != (T, d) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous [T, d] {x.dtype} tensor")
    rc = load_library().gelu_and_mul_sparse_native(out.data_ptr(), x.data_ptr(), T, d, rs,
                                                   float(z), _DTYPE_CODE[x.dtype],
                                                   _stream_handle(stream))
    _check("gelu_and_mul_sparse_native", rc)
    return out


def gelu_and_mul_sparse_plan(x: torch.Tensor, d: int | None = None, out: torch.Tensor | None = None,
                             variant: int = VARIANT_AUTO, cluster: int = 0,
                             workspace: bool = False) -> dict:
    """The launch geometry gelu_and_mul_sparse would use for this call
    (``workspace``: a call that passes a workspace)."""
    T, rs = _rows_view(x, tuple(_DTYPE_CODE))
    d = int(x.shape[1]) // 2 if d is None else d
    p = Plan()
    out_ptr = out.data_ptr() if out is not None else 0
    rc = load_library().gelu_and_mul_sparse_plan_ex(out_ptr, x.data_ptr(), T, d, rs,
                                                    _DTYPE_CODE[x.dtype], int(variant),
                                                    int(cluster), 0, int(bool(workspace)),
                                                    ctypes.byref(p))
    _check("gelu_and_mul_sparse_plan", rc)
    return p.as_dict()


def gelu_and_mul_sparse_native_plan(x: torch.Tensor, d: int | None = None) -> dict:
    """The launch geometry gelu_and_mul_sparse_native would use for ``x``."""
    T, rs = _rows_view(x, (torch.bfloat16, torch.float16))
    d = int(x.shape[1]) // 2 if d is None else d
    p = Plan()
    rc = load_library().gelu_and_mul_sparse_native_plan(0, x.data_ptr(), T, d, rs,
                                                        _DTYPE_CODE[x.dtype], 0, ctypes.byref(p))
    _check("gelu_and_mul_sparse_native_plan", rc)
    return p.as_dict()


def device_status() -> int:
    """Status bits the library's kernels raised on the current device (then cleared).

    Bit 0: a bounded wait for a bulk copy gave up.  Synchronizes the device.
    """
    v = ctypes.c_uint(0)
    _check("gated_act_device_status", load_library().gated_act_device_status(ctypes.byref(v)))
    return int(v.value)


def noop(stream: torch.cuda.Stream | None = None) -> None:
    """Launch the library's empty kernel (launch-overhead probe)."""
    _check("gated_act_noop", load_library().gated_act_noop(_stream_handle(stream)))


def silu_and_mul(x: torch.Tensor, out: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """silu(gate) * up of a contiguous [M, 2d] bf16 tensor (CUDA or page-locked
    host): returns [M, d] bf16 where x lives."""
    if x.dim() != 2 or x.dtype != torch.bfloat16 or not _is_device_or_pinned(x) \
            or not x.is_contiguous():
        raise ValueError("input must be a contiguous 2-D bf16 tensor [M, 2d] on the device "
                         "or in page-locked host memory")
    M, w = int(x.shape[0]), int(x.shape[1])
    if w % 2:
        raise ValueError("row length must be even (2d)")
    d = w // 2
    if out is None:
        out = _empty_like_rows(x, M, d)
    elif out.shape != (M, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, d] bf16 tensor")
    rc = load_library().silu_and_mul(out.data_ptr(), x.data_ptr(), M, d, _stream_handle(stream))
    _check("silu_and_mul", rc)
    return out


def _gated_in(x: torch.Tensor, d: int | None) -> tuple[int, int, int]:
    T, rs = _rows_view(x)
    if d is None:
        if x.shape[1] % 2:
            raise ValueError("odd row length: pass d explicitly")
        d = int(x.shape[1]) // 2
    if x.shape[1] < 2 * d:
        raise ValueError("rows are shorter than 2d")
    return T, rs, d


def _out_for(out: torch.Tensor | None, T: int, d: int, like: torch.Tensor) -> torch.Tensor:
    if out is None:
        return _empty_like_rows(like, T, d)
    if out.shape != (T, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous [{T}, {d}] bf16 tensor")
    return out


def silu_and_mul_bounded(x: torch.Tensor, n_rows: torch.Tensor, out: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """silu_and_mul over the first ``n_rows`` rows (a 1-element int32 tensor).

    Rows at or past the live count are left untouched in ``out``.
    """
    if x.dim() != 2 or x.dtype != torch.bfloat16 or not _is_device_or_pinned(x) \
            or not x.is_contiguous():
        raise ValueError("input must be a contiguous 2-D bf16 tensor [M, 2d]")
    if n_rows.dtype != torch.int32 or not _is_device_or_pinned(n_rows) or n_rows.numel() < 1:
        raise ValueError("n_rows must be an int32 tensor on the device or in page-locked memory")
    M, d = int(x.shape[0]), int(x.shape[1]) // 2
    out = _out_for(out, M, d, x)
    rc = load_library().silu_and_mul_bounded(out.data_ptr(), x.data_ptr(), M, d,
                                             n_rows.data_ptr(), _stream_handle(stream))
    _check("silu_and_mul_bounded", rc)
    return out


def gelu_and_mul(x: torch.Tensor, d: int | None = None, out: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Dense gelu_tanh(gate) * up of ``x`` ([T, >=2d] bf16): returns [T, d] bf16."""
    T, rs, d = _gated_in(x, d)
    out = _out_for(out, T, d, x)
    rc = load_library().gelu_and_mul(out.data_ptr(), x.data_ptr(), T, d, rs, _stream_handle(stream))
    _check("gelu_and_mul", rc)
    return out


def squared_relu(x: torch.Tensor, out: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """max(x, 0)^2 of a contiguous [M, d] bf16 tensor."""
    if x.dim() != 2 or x.dtype != torch.bfloat16 or not _is_device_or_pinned(x) \
            or not x.is_contiguous():
        raise ValueError("input must be a contiguous 2-D bf16 tensor [M, d]")
    M, d = int(x.shape[0]), int(x.shape[1])
    out = _out_for(out, M, d, x)
    rc = load_library().squared_relu(out.data_ptr(), x.data_ptr(), M, d, _stream_handle(stream))
    _check("squared_relu", rc)
    return out


__all__ = ["gelu_and_mul_sparse_native", "gelu_and_mul_sparse_native_plan", "silu_and_mul_bounded", "gelu_and_mul", "squared_relu", "gelu_and_mul_sparse", "gelu_and_mul_sparse_plan", "silu_and_mul", "device_status", "noop",
           "load_library",
           "status_string", "GatedActError", "Plan", "EXPORTED", "LIB_PATH", "workspace_bytes",
           "new_workspace"]
