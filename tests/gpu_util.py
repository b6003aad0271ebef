"""Shared set-up for the GPU tests: the device, the built library, guarded buffers."""
from __future__ import annotations

import pytest
import torch

SENTINEL = 0x7FA1          # a NaN bit pattern no kernel writes
GUARD = 64                 # elements of guard band on each side (128 B keeps 16-byte alignment)


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_activation_gb300 as ga
    from gated_activation_gb300 import build as gbuild
    if not gbuild.up_to_date():
        gbuild.build()
    return ga


def guarded_empty(shape, device="cuda"):
    """bf16 tensor of `shape` inside a buffer whose guard bands hold SENTINEL."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.int16, device=device)
    out = buf[GUARD:GUARD + n].view(torch.bfloat16).view(*shape)
    return buf, out


def guards_intact(buf) -> bool:
    head = buf[:GUARD]
    tail = buf[buf.numel() - GUARD:]
    return bool((head == SENTINEL).all().item() and (tail == SENTINEL).all().item())
