"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and lays them out; it holds none of the
activation's arithmetic.  Every tensor is drawn on the CPU from
``torch.Generator().manual_seed(seed)`` in float32 and then rounded to bf16,
so both the CUDA path and the oracle see the same bits.

The recipes stand in for the activations that the pages' model runs produced
(Gemma3n decode/prefill for the sparse GELU, Qwen3-30B-A3B MoE decode for
silu_and_mul); none of those tensors exist here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

# z = inverse standard-normal CDF at the target sparsity 0.95.
Z95 = 1.6448536269514722

SWEEP_T = (1, 8, 64, 256, 1024, 2048)
SWEEP_D = (2048, 4096, 8192, 16384, 32768)
SWEEP_Z = (0.0, Z95)
DECODE_T = (1, 2, 4, 8, 16, 32, 64)
DECODE_D = 8192
PREFILL_T, PREFILL_D = 2048, 16384
TINY_T, TINY_D = 4, 2048
SILU_D = 768
SILU_M = (1024, 2048, 4096, 16384)
CONST_GATES = (0.0, 0.75, -1.25)   # exactly representable in bf16


@dataclass
class GatedInput:
    """One [T, row_stride] bf16 input: gate = [:, :d], up = [:, d:2d]."""

    name: str
    x: torch.Tensor        # CPU bf16, shape [T, row_stride]
    d: int
    z: float
    seed: int

    @property
    def T(self) -> int:
        return int(self.x.shape[0])

    @property
    def row_stride(self) -> int:
        return int(self.x.shape[1])


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def to_bits(x: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (no copy of values)."""
    assert x.dtype == torch.bfloat16
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def iid(T: int, d: int, seed: int, row_stride: int | None = None,
        z: float = Z95, name: str = "iid", pad_value: float = math.nan,
        dtype: torch.dtype = torch.bfloat16) -> GatedInput:
    """Gate and up i.i.d. N(0,1), drawn as one [T, 2d] tensor.

    With ``row_stride > 2d`` the extra columns hold ``pad_value`` (NaN by
    default) so that a stray read of padding poisons the output.  ``dtype``
    is the element type the float32 draws are rounded to (once).
    """
    g = _gen(seed)
    x = torch.randn((T, 2 * d), generator=g, dtype=torch.float32)
    return GatedInput(name, _pad(x, row_stride, pad_value, dtype), d, z, seed)


def _pad(x: torch.Tensor, row_stride: int | None, pad_value: float,
         dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    T, w = x.shape
    if row_stride is None or row_stride == w:
        return x.to(dtype)
    if row_stride < w:
        raise ValueError("row_stride must be >= 2d")
    out = torch.full((T, row_stride), pad_value, dtype=torch.float32)
    out[:, :w] = x
    return out.to(dtype)


def tiny() -> GatedInput:
    """T=4, d=2048, [4, 4096] contiguous, i.i.d. N(0,1), seed 0, z for 0.95."""
    return iid(TINY_T, TINY_D, seed=0, name="tiny")


def decode(T: int, d: int = DECODE_D, dtype: torch.dtype = torch.bfloat16) -> GatedInput:
    """Decode rows: d=8192, seed 1000+T.

    gate = 0.2 + 1.5 * N(0,1); each gate entry is independently (probability
    0.01) replaced by an outlier 8 * N(0,1); up = N(0,1).  Draw order: gate
    base, outlier selector (uniform), outlier values, up.
    """
    seed = 1000 + T
    g = _gen(seed)
    gate = 0.2 + 1.5 * torch.randn((T, d), generator=g)
    sel = torch.rand((T, d), generator=g) < 0.01
    outl = 8.0 * torch.randn((T, d), generator=g)
    gate = torch.where(sel, outl, gate)
    up = torch.randn((T, d), generator=g)
    x = torch.cat([gate, up], dim=1).to(dtype)
    return GatedInput(f"decode_T{T}", x, d, Z95, seed)


def prefill(T: int = PREFILL_T, d: int = PREFILL_D,
            dtype: torch.dtype = torch.bfloat16) -> GatedInput:
    """Prefill rows: T=2048, d=16384, row_stride 32768 = 2d, seed 2.

    gate = s_r * N(0,1) + m_r with per-row scale s_r ~ U(0.5, 2) and shift
    m_r ~ U(-1, 1); up = N(0,1).  Draw order: s, m, gate noise, up.
    """
    seed = 2
    g = _gen(seed)
    s = 0.5 + 1.5 * torch.rand((T, 1), generator=g)
    m = -1.0 + 2.0 * torch.rand((T, 1), generator=g)
    gate = s * torch.randn((T, d), generator=g) + m
    up = torch.randn((T, d), generator=g)
    x = torch.cat([gate, up], dim=1).to(dtype)
    return GatedInput("prefill", x, d, Z95, seed)


def sweep_seed(T: int, d: int) -> int:
    return 7919 * T + d


def sweep(T: int, d: int, z: float = Z95, const_rows: bool = True,
          dtype: torch.dtype = torch.bfloat16) -> GatedInput:
    """Sweep shape (T, d): i.i.d. N(0,1), seed 7919*T + d.

    With ``const_rows`` three rows whose gate is all one constant (0, 0.75,
    -1.25; std = 0) are appended after the T random rows, their up halves
    N(0,1) from the same generator: the correctness input is [T+3, 2d], the
    timed input exactly the first T rows.
    """
    seed = sweep_seed(T, d)
    g = _gen(seed)
    x = torch.randn((T, 2 * d), generator=g, dtype=torch.float32)
    if const_rows:
        up = torch.randn((len(CONST_GATES), d), generator=g)
        gate = torch.tensor(CONST_GATES, dtype=torch.float32)[:, None].expand(-1, d)
        x = torch.cat([x, torch.cat([gate, up], dim=1)], dim=0)
    return GatedInput(f"sweep_T{T}_d{d}", x.to(dtype), d, z, seed)


def silu(M: int, d: int = SILU_D) -> torch.Tensor:
    """MoE decode rows for silu_and_mul: [M, 2d] contiguous, i.i.d. N(0,1), seed 3+M."""
    g = _gen(3 + M)
    return torch.randn((M, 2 * d), generator=g).to(torch.bfloat16)


__all__ = [
    "Z95", "SWEEP_T", "SWEEP_D", "SWEEP_Z", "DECODE_T", "DECODE_D", "PREFILL_T",
    "PREFILL_D", "TINY_T", "TINY_D", "SILU_D", "SILU_M", "CONST_GATES", "GatedInput",
    "to_bits", "from_bits", "iid", "tiny", "decode", "prefill", "sweep", "sweep_seed",
    "silu",
]
