"""GPU parity of gelu_and_mul_sparse's native-rounding mode (bf16, fp16)
against the native-rounding oracle, and against PyTorch's own CUDA
composition of the separate ops -- the behaviour this mode reproduces
(sparse-GELU page, "Cross-architecture warp and dtype validation")."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_native

pytestmark = pytest.mark.gpu
DTYPES = [torch.bfloat16, torch.float16]


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def oracle_native(oracle, x, d, z):
    arr = W.to_bits(x.contiguous()) if x.dtype == torch.bfloat16 else x.contiguous().numpy()
    return oracle.gelu_and_mul_sparse_native(arr, d=d, z=z, bf16_bits=x.dtype == torch.bfloat16)


def run(ga, x, d, z):
    out = ga.gelu_and_mul_sparse_native(x.cuda(), z, d=d)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("z", [W.Z95, 0.0, 1.3])
@pytest.mark.parametrize("dt", DTYPES)
def test_native_against_oracle(ga, oracle, dt, z):
    for inp in (W.iid(4, 2048, seed=0, dtype=dt), W.decode(8, dtype=dt),
                W.prefill(T=512, dtype=dt), W.sweep(64, 32768, z=z, dtype=dt)):
        ref, mask, cut = oracle_native(oracle, inp.x, inp.d, z)
        check_native(run(ga, inp.x, inp.d, z), inp.x, inp.d, ref, mask, cut,
                     f"{dt} {inp.name} z{z}", z=z)


@pytest.mark.parametrize("dt", DTYPES)
def test_native_constant_rows_and_ragged(ga, oracle, dt):
    inp = W.sweep(8, 2048, dtype=dt)
    ref, mask, cut = oracle_native(oracle, inp.x, 2048, inp.z)
    out = run(ga, inp.x, 2048, inp.z)
    check_native(out, inp.x, 2048, ref, mask, cut, f"{dt} const", z=inp.z)
    assert torch.count_nonzero(out[-3:].float()).item() == 0
    for T, d, rs in ((5, 31, None), (3, 1, None), (4, 1000, 2048 + 8)):
        inp = W.iid(T, d, seed=d, row_stride=rs, dtype=dt)
        ref, mask, cut = oracle_native(oracle, inp.x, d, inp.z)
        check_native(run(ga, inp.x, d, inp.z), inp.x, d, ref, mask, cut, f"{dt} d{d}", z=inp.z)


@pytest.mark.parametrize("dt", DTYPES)
def test_native_reproduces_torch_cuda_composition(ga, dt):
    # PyTorch's own composition of separate element-type ops on the GPU: the
    # native mode must give the same zero pattern and values except on the
    # rare rows whose fp32 statistics round differently in the two reductions
    inp = W.prefill(T=1024, dtype=dt)
    x = inp.x.cuda()
    d = inp.d
    g, u = x[:, :d], x[:, d:]
    c = g.mean(dim=1, keepdim=True) + g.std(dim=1, keepdim=True, unbiased=False) * inp.z
    want = F.gelu(torch.relu(g - c), approximate="tanh") * u
    got = ga.gelu_and_mul_sparse_native(x, inp.z)
    torch.cuda.synchronize()
    same_rows = (got.view(torch.int16) == want.view(torch.int16)).all(dim=1).float().mean().item()
    mask_mismatch = ((got != 0) != (want != 0)).float().mean().item()
    assert same_rows >= 0.95, same_rows
    assert mask_mismatch <= 1e-4, mask_mismatch


def test_native_rejects_fp32(ga):
    x = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        ga.gelu_and_mul_sparse_native(x, 1.0)
