"""GPU parity of gelu_and_mul_sparse on fp16 and fp32 rows (the sparse-GELU
page validates FP32, FP16 and BF16), through the C ABI, against the fp64
oracle with per-type tolerances (tests/parity.py TOLERANCES)."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu
DTYPES = [torch.float16, torch.float32]


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def oracle_typed(oracle, x, d, z):
    return oracle.gelu_and_mul_sparse_typed(x.contiguous().numpy(), d=d, z=z)


def run(ga, x, d, z, **kw):
    out = ga.gelu_and_mul_sparse(x.cuda(), z, d=d, **kw)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("dt", DTYPES)
def test_typed_tiny_decode_prefill(ga, oracle, dt):
    for inp in (W.iid(4, 2048, seed=0, dtype=dt), W.decode(1, dtype=dt), W.decode(64, dtype=dt),
                W.prefill(dtype=dt)):
        res = oracle_typed(oracle, inp.x, inp.d, inp.z)
        check_gelu(run(ga, inp.x, inp.d, inp.z), inp.x, inp.d, res, f"{dt} {inp.name}")


@pytest.mark.parametrize("z", W.SWEEP_Z)
@pytest.mark.parametrize("T,d", [(1, 2048), (8, 32768), (64, 4096), (256, 8192), (1024, 16384),
                                 (2048, 32768)])
@pytest.mark.parametrize("dt", DTYPES)
def test_typed_sweep_with_constant_rows(ga, oracle, dt, T, d, z):
    inp = W.sweep(T, d, z=z, const_rows=True, dtype=dt)
    res = oracle_typed(oracle, inp.x, d, z)
    out = run(ga, inp.x, d, z)
    check_gelu(out, inp.x, d, res, f"{dt} sweep T{T} d{d} z{z}")
    assert torch.count_nonzero(out[-3:].float()).item() == 0


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("dt", DTYPES)
def test_typed_forced_clusters(ga, oracle, dt, cluster):
    inp = W.iid(16, 16384, seed=5, dtype=dt)
    res = oracle_typed(oracle, inp.x, 16384, inp.z)
    check_gelu(run(ga, inp.x, 16384, inp.z, variant=2, cluster=cluster), inp.x, 16384, res,
               f"{dt} c{cluster}")


@pytest.mark.parametrize("T,d,rs", [(5, 1, None), (7, 3, None), (4, 31, None), (3, 6, None),
                                    (6, 12, None), (9, 1000, 2048 + 8), (4, 2048, 4099),
                                    (3, 65536, None)])
@pytest.mark.parametrize("dt", DTYPES)
def test_typed_ragged_strided_wide(ga, oracle, dt, T, d, rs):
    inp = W.iid(T, d, seed=T + d, row_stride=rs, dtype=dt)
    res = oracle_typed(oracle, inp.x, d, inp.z)
    check_gelu(run(ga, inp.x, d, inp.z), inp.x, d, res, f"{dt} T{T} d{d} rs{rs}")


@pytest.mark.parametrize("dt", DTYPES)
def test_typed_misaligned_pointer_and_nan(ga, oracle, dt):
    T, d = 6, 1024
    inp = W.iid(T, d, seed=2, dtype=dt)
    x = inp.x.clone()
    x[2, 10] = float("nan")
    big = torch.zeros((T * 2 * d + 8,), dtype=dt, device="cuda")
    big[1:1 + T * 2 * d] = x.reshape(-1).cuda()
    out = ga.gelu_and_mul_sparse(big[1:1 + T * 2 * d].view(T, 2 * d), inp.z)
    torch.cuda.synchronize()
    res = oracle_typed(oracle, x, d, inp.z)
    check_gelu(out.cpu(), x, d, res, f"{dt} misaligned")
    assert torch.isnan(out[2].float()).all()


@pytest.mark.parametrize("dt", DTYPES)
def test_typed_same_values_as_bf16_within_tolerance(ga, dt):
    # bf16 values carried in a wider type: both paths see the same numbers
    inp = W.iid(64, 8192, seed=3)
    a = ga.gelu_and_mul_sparse(inp.x.cuda(), inp.z).float()
    b = ga.gelu_and_mul_sparse(inp.x.to(dt).cuda(), inp.z).float()
    torch.cuda.synchronize()
    assert torch.allclose(a, b, rtol=1e-2, atol=2e-3)
