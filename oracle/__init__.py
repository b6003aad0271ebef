"""fp64 CPU oracle for the fused gated activations -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never do, and nothing here calls them.

The arithmetic lives in ``gated_act_oracle.c`` (plain fp64 C, one loop per
stage); this module only loads the compiled library and marshals numpy arrays.
Inputs are bf16 bit patterns as ``numpy.uint16`` arrays.

  gelu_and_mul_sparse -- vLLM PR "[Performance] Add Triton kernel for Gemma3n
      sparse GELU", section "Purpose" (per-row mean and variance, Gaussian
      thresholding, tanh GELU, gated multiplication).
  silu_and_mul -- Megatron-LM PR "Size MoE activation kernel grid to the row
      count", section "What changed and why" (elementwise silu(gate) * up).
  squared_relu -- same page, section "Scope and risks" (max(x, 0)^2).
  gelu_and_mul -- the dense form of the sparse-GELU activation (no threshold).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from .build import LIB, ensure_built

_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_u8_p = ctypes.POINTER(ctypes.c_uint8)
_c_u16_p = ctypes.POINTER(ctypes.c_uint16)


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctype)


@dataclass
class GeluSparseResult:
    """Oracle outputs for one gelu_and_mul_sparse call (all fp64 / bool)."""

    ref: np.ndarray      # [T, d] float64, unrounded gelu_tanh(relu(g - cutoff)) * u
    mask: np.ndarray     # [T, d] bool, g > cutoff
    mean: np.ndarray     # [T] float64
    std: np.ndarray      # [T] float64, population std
    cutoff: np.ndarray   # [T] float64, mean + std * z


class Oracle:
    """Handle on one compiled oracle library (the default one, or a variant)."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = ensure_built()
        self.path = os.path.abspath(lib_path)
        lib = ctypes.CDLL(self.path)
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_gelu_tanh.restype = ctypes.c_double
        lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_gelu_and_mul_sparse.restype = ctypes.c_int
        lib.oracle_gelu_and_mul_sparse.argtypes = [
            _c_u16_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
            _c_double_p, _c_u8_p, _c_double_p, _c_double_p, _c_double_p, ctypes.c_int]
        lib.oracle_silu_and_mul.restype = ctypes.c_int
        lib.oracle_silu_and_mul.argtypes = [
            _c_u16_p, ctypes.c_int64, ctypes.c_int64, _c_double_p, _c_u16_p, ctypes.c_int]
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_gelu_and_mul_sparse_typed.restype = ctypes.c_int
        lib.oracle_gelu_and_mul_sparse_typed.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_double, _c_double_p, _c_u8_p, _c_double_p, _c_double_p, _c_double_p,
            ctypes.c_int]
        lib.oracle_round_f16.restype = ctypes.c_double
        lib.oracle_round_f16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_double
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_gelu_and_mul_sparse_native.restype = ctypes.c_int
        lib.oracle_gelu_and_mul_sparse_native.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_double, _c_double_p, _c_u8_p, _c_double_p, ctypes.c_int]
        lib.oracle_squared_relu.restype = ctypes.c_double
        lib.oracle_squared_relu.argtypes = [ctypes.c_double]
        lib.oracle_gelu_and_mul.restype = ctypes.c_int
        lib.oracle_gelu_and_mul.argtypes = [
            _c_u16_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _c_double_p, _c_u16_p,
            ctypes.c_int]
        lib.oracle_squared_relu_rows.restype = ctypes.c_int
        lib.oracle_squared_relu_rows.argtypes = [
            _c_u16_p, ctypes.c_int64, ctypes.c_int64, _c_double_p, _c_u16_p, ctypes.c_int]
        self._lib = lib

    # -- scalar helpers -------------------------------------------------------
    def bf16_to_double(self, bits: int) -> float:
        return self._lib.oracle_bf16_to_double(int(bits) & 0xFFFF)

    def double_to_bf16(self, v: float) -> int:
        return int(self._lib.oracle_double_to_bf16(float(v)))

    def f16_to_double(self, bits: int) -> float:
        return self._lib.oracle_f16_to_double(int(bits) & 0xFFFF)

    def gelu_tanh(self, x: float) -> float:
        return self._lib.oracle_gelu_tanh(float(x))

    def silu(self, x: float) -> float:
        return self._lib.oracle_silu(float(x))

    def squared_relu(self, x: float) -> float:
        return self._lib.oracle_squared_relu(float(x))

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    # -- the two operations -----------------------------------------------------
    def gelu_and_mul_sparse(self, in_bits: np.ndarray, d: int, z: float,
                            row_stride: int | None = None,
                            nthreads: int = 0) -> GeluSparseResult:
        """Oracle for gelu_and_mul_sparse on ``in_bits`` ([T, row_stride] uint16)."""
        a = np.ascontiguousarray(in_bits, dtype=np.uint16)
        if a.ndim != 2:
            raise ValueError("in_bits must be 2-D [T, row_stride]")
        T, rs = a.shape
        if row_stride is not None and row_stride != rs:
            raise ValueError("row_stride must equal the array's row length")
        ref = np.empty((T, d), dtype=np.float64)
        mask = np.empty((T, d), dtype=np.uint8)
        mean = np.empty(T, dtype=np.float64)
        std = np.empty(T, dtype=np.float64)
        cutoff = np.empty(T, dtype=np.float64)
        rc = self._lib.oracle_gelu_and_mul_sparse(
            _ptr(a, _c_u16_p), T, d, rs, float(z), _ptr(ref, _c_double_p),
            _ptr(mask, _c_u8_p), _ptr(mean, _c_double_p), _ptr(std, _c_double_p),
            _ptr(cutoff, _c_double_p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_gelu_and_mul_sparse rejected T={T} d={d} rs={rs}")
        return GeluSparseResult(ref, mask.astype(bool), mean, std, cutoff)

    def gelu_and_mul_sparse_typed(self, x: np.ndarray, d: int, z: float,
                                  bf16_bits: bool = False, nthreads: int = 0) -> GeluSparseResult:
        """gelu_and_mul_sparse on a [T, row_stride] numpy array of float16 or
        float32 values, or of bf16 bit patterns (uint16 with bf16_bits=True)."""
        a = np.ascontiguousarray(x)
        if a.dtype == np.uint16:
            if not bf16_bits:
                raise ValueError("uint16 input must be bf16 bit patterns (bf16_bits=True)")
            code = 0
        elif a.dtype == np.float16:
            code = 1
        elif a.dtype == np.float32:
            code = 2
        else:
            raise ValueError(f"unsupported element type {a.dtype}")
        T, rs = a.shape
        ref = np.empty((T, d), dtype=np.float64)
        mask = np.empty((T, d), dtype=np.uint8)
        mean = np.empty(T, dtype=np.float64)
        std = np.empty(T, dtype=np.float64)
        cutoff = np.empty(T, dtype=np.float64)
        rc = self._lib.oracle_gelu_and_mul_sparse_typed(
            a.ctypes.data_as(ctypes.c_void_p), code, T, d, rs, float(z), _ptr(ref, _c_double_p),
            _ptr(mask, _c_u8_p), _ptr(mean, _c_double_p), _ptr(std, _c_double_p),
            _ptr(cutoff, _c_double_p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_gelu_and_mul_sparse_typed rejected T={T} d={d} rs={rs}")
        return GeluSparseResult(ref, mask.astype(bool), mean, std, cutoff)

    def round_f16(self, v: float) -> float:
        return self._lib.oracle_round_f16(float(v))

    def round_bf16(self, v: float) -> float:
        return self._lib.oracle_round_bf16(float(v))

    def gelu_and_mul_sparse_native(self, x: np.ndarray, d: int, z: float, bf16_bits: bool = False,
                                   nthreads: int = 0) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """Native-rounding gelu_and_mul_sparse on bf16 bit patterns (uint16 with
        bf16_bits=True) or float16 values.  Returns (out already rounded to the
        element type, as float64 [T, d]; mask g > c [T, d]; cutoff c [T])."""
        a = np.ascontiguousarray(x)
        if a.dtype == np.uint16 and bf16_bits:
            code = 0
        elif a.dtype == np.float16:
            code = 1
        else:
            raise ValueError("native rounding takes bf16 bit patterns or float16 values")
        T, rs = a.shape
        ref = np.empty((T, d), dtype=np.float64)
        mask = np.empty((T, d), dtype=np.uint8)
        cutoff = np.empty(T, dtype=np.float64)
        rc = self._lib.oracle_gelu_and_mul_sparse_native(
            a.ctypes.data_as(ctypes.c_void_p), code, T, d, rs, float(z), _ptr(ref, _c_double_p),
            _ptr(mask, _c_u8_p), _ptr(cutoff, _c_double_p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_gelu_and_mul_sparse_native rejected T={T} d={d} rs={rs}")
        return ref, mask.astype(bool), cutoff

    def silu_and_mul(self, in_bits: np.ndarray, d: int | None = None,
                     nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """Oracle for silu_and_mul on ``in_bits`` ([M, 2d] uint16).

        Returns (ref fp64 [M, d], ref rounded to bf16 bits uint16 [M, d]).
        """
        a = np.ascontiguousarray(in_bits, dtype=np.uint16)
        M, w = a.shape
        if d is None:
            d = w // 2
        if w != 2 * d:
            raise ValueError("silu_and_mul input must be contiguous [M, 2d]")
        ref = np.empty((M, d), dtype=np.float64)
        ref16 = np.empty((M, d), dtype=np.uint16)
        rc = self._lib.oracle_silu_and_mul(_ptr(a, _c_u16_p), M, d,
                                           _ptr(ref, _c_double_p),
                                           _ptr(ref16, _c_u16_p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_silu_and_mul rejected M={M} d={d}")
        return ref, ref16


    def gelu_and_mul(self, in_bits: np.ndarray, d: int, row_stride: int | None = None,
                     nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """Dense gelu_tanh(g) * u on ``in_bits`` ([T, row_stride] uint16).

        Returns (ref fp64 [T, d], ref rounded to bf16 bits uint16 [T, d]).
        """
        a = np.ascontiguousarray(in_bits, dtype=np.uint16)
        T, rs = a.shape
        if row_stride is not None and row_stride != rs:
            raise ValueError("row_stride must equal the array's row length")
        ref = np.empty((T, d), dtype=np.float64)
        ref16 = np.empty((T, d), dtype=np.uint16)
        rc = self._lib.oracle_gelu_and_mul(_ptr(a, _c_u16_p), T, d, rs, _ptr(ref, _c_double_p),
                                           _ptr(ref16, _c_u16_p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_gelu_and_mul rejected T={T} d={d} rs={rs}")
        return ref, ref16

    def squared_relu_rows(self, in_bits: np.ndarray,
                          nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """max(x, 0)^2 on ``in_bits`` ([M, d] uint16): (ref fp64, ref bf16 bits)."""
        a = np.ascontiguousarray(in_bits, dtype=np.uint16)
        M, d = a.shape
        ref = np.empty((M, d), dtype=np.float64)
        ref16 = np.empty((M, d), dtype=np.uint16)
        rc = self._lib.oracle_squared_relu_rows(_ptr(a, _c_u16_p), M, d, _ptr(ref, _c_double_p),
                                                _ptr(ref16, _c_u16_p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_squared_relu_rows rejected M={M} d={d}")
        return ref, ref16


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``gated_act_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


__all__ = ["Oracle", "GeluSparseResult", "default", "LIB", "ensure_built"]
