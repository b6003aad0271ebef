"""The native-rounding acceptance check itself (CPU): a row whose exact
population std lies next to a midpoint between two fp16 values may take
either rounding; a row that is not next to one may not."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as W
from tests.parity import _stat_roundings, check_native

D, Z = 520, 1.3


def _rows():
    # a seeded fp16 draw in which row 899's exact std lies 1.5 fp32 ulps from
    # the midpoint between two fp16 values
    x = W.iid(1141, D, seed=570329, row_stride=2 * D, z=Z, dtype=torch.float16).x
    return x[[899, 0]].contiguous()


def _composition(row: torch.Tensor, m: float, s: float) -> torch.Tensor:
    """PyTorch's CPU composition of the native ops with the given rounded statistics."""
    c = torch.tensor(m, dtype=row.dtype) + torch.tensor(s, dtype=row.dtype) * Z
    return F.gelu(torch.relu(row[:D] - c), approximate="tanh") * row[D:2 * D]


def _stats(row: torch.Tensor):
    g = row[:D].to(torch.float64).numpy()
    m = float(g.mean())
    s = float(np.sqrt(((g - m) ** 2).mean()))
    return (_stat_roundings(m, 2.0 ** -24 * float(np.abs(g).sum()), torch.float16),
            _stat_roundings(s, 2.0 ** -24 * (D / 2 + 2) * s, torch.float16))


def test_ambiguous_row_accepts_the_other_rounding(oracle):
    x = _rows()
    ref, mask, cut = oracle.gelu_and_mul_sparse_native(x.numpy(), d=D, z=Z, bf16_bits=False)
    ms, ss = _stats(x[0])
    assert len(ss) == 2, "row 899's std should be next to a midpoint"
    out = torch.from_numpy(ref).to(torch.float16)
    assert check_native(out, x, D, ref, mask, cut, "oracle", z=Z)["rows_other_rounding"] == 0
    alt = out.clone()
    alt[0] = _composition(x[0], ms[0], ss[1])
    assert not torch.equal(alt[0], out[0])
    assert check_native(alt, x, D, ref, mask, cut, "other rounding", z=Z)["rows_other_rounding"] == 1
    with pytest.raises(AssertionError):
        check_native(alt, x, D, ref, mask, cut, "no z")


def test_unambiguous_row_rejects_another_rounding(oracle):
    # gates shifted by 2 keep the mean away from zero, so the summation bound
    # is far below half an fp16 step; take the first such row that is clear of
    # every midpoint in both statistics
    x = W.iid(64, D, seed=570329, row_stride=2 * D, z=Z, dtype=torch.float16).x.clone()
    x[:, :D] += 2.0
    pick = next(r for r in range(x.shape[0]) if all(len(v) == 1 for v in _stats(x[r])))
    x = x[[pick]].contiguous()
    ref, mask, cut = oracle.gelu_and_mul_sparse_native(x.numpy(), d=D, z=Z, bf16_bits=False)
    (m,), (s,) = _stats(x[0])
    bad = torch.from_numpy(ref).to(torch.float16)
    for side in (1, -1):
        other = float(torch.tensor(s, dtype=torch.float16).view(torch.int16).add(side)
                      .view(torch.float16))
        bad[0] = _composition(x[0], m, other)
        assert not torch.equal(bad[0], torch.from_numpy(ref[0]).to(torch.float16))
        with pytest.raises(AssertionError):
            check_native(bad, x, D, ref, mask, cut, "unjustified rounding", z=Z)
    good = torch.from_numpy(ref).to(torch.float16)
    assert check_native(good, x, D, ref, mask, cut, "oracle", z=Z)["rows_other_rounding"] == 0
