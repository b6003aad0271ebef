"""GPU parity of silu_and_mul against the fp64 oracle (<= 1 bf16 ulp), through the C ABI.

MoE decode rows M in {1024, 2048, 4096, 16384} at d = 768, ragged and
misaligned layouts (scalar path), bitwise agreement of the vector and scalar
paths (the math per element does not depend on the geometry), extreme gate
values, guard bands.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import guarded_empty, guards_intact, require_gpu
from tests.parity import bits_of, check_silu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


@pytest.mark.parametrize("M", W.SILU_M)
def test_moe_decode_rows(ga, oracle, M):
    x = W.silu(M)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x))
    out = ga.silu_and_mul(x.cuda())
    torch.cuda.synchronize()
    check_silu(out, ref16, f"M{M}")


@pytest.mark.parametrize("M,d", [(1, 1), (3, 7), (5, 33), (17, 768), (1, 8), (1000, 100), (2, 4100)])
def test_ragged_shapes(ga, oracle, M, d):
    g = torch.Generator().manual_seed(M * 31 + d)
    x = torch.randn((M, 2 * d), generator=g).to(torch.bfloat16)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x), d=d)
    check_silu(ga.silu_and_mul(x.cuda()), ref16, f"M{M} d{d}")


def test_vector_and_scalar_paths_agree_bitwise(ga):
    M, d = 300, 768
    x = W.silu(M, d)
    a = ga.silu_and_mul(x.cuda())
    big = torch.zeros((M * 2 * d + 8,), dtype=torch.bfloat16, device="cuda")
    big[1:1 + M * 2 * d] = x.reshape(-1).cuda()
    xm = big[1:1 + M * 2 * d].view(M, 2 * d)          # 2-byte offset: scalar path
    b = ga.silu_and_mul(xm)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_extreme_gate_values(ga, oracle):
    vals = torch.tensor([0.0, -0.0, 1.0, -1.0, 10.0, -10.0, 30.0, -30.0, 80.0, -80.0,
                         -88.0, -89.0, -95.0, -100.0, -120.0, 88.5, 1e-30, -1e-30,
                         float("inf"), float("-inf"), float("nan"), 3e38, -3e38, 0.5],
                        dtype=torch.float32)
    d = vals.numel()
    up = torch.linspace(-2, 2, d)
    x = torch.cat([vals, up]).reshape(1, 2 * d).to(torch.bfloat16)
    x = x.repeat(8, 1)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x), d=d)
    check_silu(ga.silu_and_mul(x.cuda()), ref16, "extremes")


def test_guard_bands_untouched(ga):
    for M, d in ((2048, 768), (7, 33)):
        x = W.silu(M, d)
        buf, out = guarded_empty((M, d))
        ga.silu_and_mul(x.cuda(), out=out)
        torch.cuda.synchronize()
        assert guards_intact(buf)


def test_zero_rows(ga):
    out = ga.silu_and_mul(torch.empty((0, 1536), dtype=torch.bfloat16, device="cuda"))
    assert out.shape == (0, 768)
