"""Randomised GPU parity of the elementwise activations: silu_and_mul, its
bounded form, dense gelu_and_mul and squared_relu.

Each seeded draw picks the op, the row count, the width (16-byte layouts and
any other), a misaligned start (one element into a larger buffer) and, for the
bounded silu, a live-row count from below zero to past M.  Outputs are
checked against the fp64 oracle: within one bf16 ulp (silu, dense GELU), bit
exact (squared_relu), and rows at or past the live count untouched.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import SENTINEL, require_gpu
from tests.parity import bits_of, check_silu

pytestmark = pytest.mark.gpu

# GATED_ACT_FUZZ_SCALE=k runs k times as many draws (the first ones unchanged)
N_CASES = 120 * max(1, int(os.environ.get("GATED_ACT_FUZZ_SCALE", "1")))
MAX_ELEMS = 4_000_000
OPS = ("silu", "silu_bounded", "gelu_dense", "squared_relu")


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def draw(i: int) -> dict:
    r = np.random.default_rng(40_000 + i)
    op = OPS[int(r.integers(len(OPS)))]
    if r.random() < 0.75:
        d = 8 * int(np.exp(r.uniform(0.0, np.log(4096))))
    else:
        d = int(np.exp(r.uniform(0.0, np.log(20000))))
    d = max(d, 1)
    M = max(1, int(min(MAX_ELEMS // d, np.exp(r.uniform(0.0, np.log(20000))))))
    return {"op": op, "M": M, "d": d, "offset": int(r.random() < 0.2),
            "n_rows": int(r.integers(-2, M + 3)), "seed": 50_000 + i}


def _on_device(x: torch.Tensor, offset: int) -> torch.Tensor:
    """x on the device, starting `offset` elements into a larger buffer."""
    flat = torch.empty(x.numel() + 8, dtype=x.dtype, device="cuda")
    flat[offset:offset + x.numel()] = x.reshape(-1).cuda()
    return flat[offset:offset + x.numel()].view(x.shape)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_elementwise(ga, oracle, i):
    c = draw(i)
    M, d, op = c["M"], c["d"], c["op"]
    g = torch.Generator().manual_seed(c["seed"])
    width = d if op == "squared_relu" else 2 * d
    x = (2.5 * torch.randn((M, width), generator=g)).to(torch.bfloat16)
    xd = _on_device(x, c["offset"])
    label = f"case {i}: {c}"
    if op == "squared_relu":
        _, ref16 = oracle.squared_relu_rows(W.to_bits(x))
        got = bits_of(ga.squared_relu(xd))
        same = (got == ref16) | (((got | ref16) & 0x7FFF) == 0)
        assert same.all(), label
        return
    if op == "gelu_dense":
        _, ref16 = oracle.gelu_and_mul(W.to_bits(x), d=d)
        check_silu(ga.gelu_and_mul(xd, d=d), ref16, label)
        return
    _, ref16 = oracle.silu_and_mul(W.to_bits(x), d=d)
    if op == "silu":
        check_silu(ga.silu_and_mul(xd), ref16, label)
        return
    live = min(max(c["n_rows"], 0), M)
    out = torch.full((M, d), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL)
    out = out.view(torch.bfloat16)
    nr = torch.tensor([c["n_rows"]], dtype=torch.int32, device="cuda")
    ga.silu_and_mul_bounded(xd, nr, out=out)
    torch.cuda.synchronize()
    if live:
        check_silu(out[:live], ref16[:live], label)
    assert (out[live:].view(torch.int16) == SENTINEL).all().item(), label
