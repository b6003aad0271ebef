"""Host buffers: page-locked host memory passed straight to the C ABI is read
and written by the kernels in place (over the CPU-GPU link).  Results must
match the oracle exactly as device buffers do."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import SENTINEL, require_gpu
from tests.parity import check_gelu, check_silu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


# (16, 16384): device buffers would take split rows, which host memory refuses
@pytest.mark.parametrize("T,d", [(4, 2048), (64, 8192), (2048, 16384), (3, 32768), (5, 31),
                                 (16, 16384)])
def test_gelu_on_pinned_host_buffers(ga, oracle, T, d):
    inp = W.iid(T, d, seed=T + d)
    x = inp.x.pin_memory()
    out = ga.gelu_and_mul_sparse(x, inp.z)
    torch.cuda.synchronize()
    assert not out.is_cuda and out.is_pinned()
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    check_gelu(out, inp.x, d, res, f"host T{T} d{d}")
    plan = ga.gelu_and_mul_sparse_plan(x)           # a plan query never sees host memory
    assert plan["variant"] in ("warp_rows", "cta_row", "tma_rows", "scalar")


def test_gelu_mixed_host_and_device(ga, oracle):
    inp = W.iid(300, 4096, seed=5)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=4096, z=inp.z)
    # device input, host output
    out_h = torch.empty((300, 4096), dtype=torch.bfloat16, pin_memory=True)
    ga.gelu_and_mul_sparse(inp.x.cuda(), inp.z, out=out_h)
    torch.cuda.synchronize()
    check_gelu(out_h, inp.x, 4096, res, "device in, host out")
    # host input, device output
    out_d = ga.gelu_and_mul_sparse(inp.x.pin_memory(), inp.z,
                                   out=torch.empty((300, 4096), dtype=torch.bfloat16,
                                                   device="cuda"))
    torch.cuda.synchronize()
    check_gelu(out_d.cpu(), inp.x, 4096, res, "host in, device out")


@pytest.mark.parametrize("variant", ["VARIANT_TMA_ROWS", "VARIANT_PIPE_ROWS"])
def test_bulk_copy_rows_refuse_host_memory(ga, variant):
    x = W.iid(400, 4096, seed=1).x.pin_memory()
    with pytest.raises(ga.GatedActError) as e:
        ga.gelu_and_mul_sparse(x, W.Z95, variant=getattr(ga, variant))
    assert e.value.status == ga.ERR_VARIANT


@pytest.mark.parametrize("dt", [torch.float16, torch.float32])
def test_typed_on_pinned_host(ga, oracle, dt):
    inp = W.iid(33, 2048, seed=9, dtype=dt)
    out = ga.gelu_and_mul_sparse(inp.x.pin_memory(), inp.z)
    torch.cuda.synchronize()
    res = oracle.gelu_and_mul_sparse_typed(inp.x.numpy(), d=2048, z=inp.z)
    check_gelu(out, inp.x, 2048, res, f"host {dt}")


def test_silu_family_on_pinned_host(ga, oracle):
    x = W.silu(2048)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x))
    xh = x.pin_memory()
    check_silu(ga.silu_and_mul(xh), ref16, "silu host")
    out = torch.empty((2048, 768), dtype=torch.bfloat16, pin_memory=True)
    out.view(torch.int16).fill_(SENTINEL)
    nr = torch.tensor([1000], dtype=torch.int32).pin_memory()   # live count in host memory too
    ga.silu_and_mul_bounded(xh, nr, out=out)
    torch.cuda.synchronize()
    check_silu(out[:1000], ref16[:1000], "bounded host")
    assert (out[1000:].view(torch.int16) == SENTINEL).all().item()
    g = torch.Generator().manual_seed(1)
    q = (3 * torch.randn((512, 768), generator=g)).to(torch.bfloat16)
    _, q16 = oracle.squared_relu_rows(W.to_bits(q))
    got = ga.squared_relu(q.pin_memory())
    torch.cuda.synchronize()
    assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), q16)


def test_pageable_memory_is_refused_before_launch(ga):
    x = W.iid(8, 2048, seed=2).x                      # ordinary (pageable) host tensor
    with pytest.raises(ValueError):
        ga.gelu_and_mul_sparse(x, W.Z95)
    out = torch.empty((8, 2048), dtype=torch.bfloat16, device="cuda")
    lib = ga.load_library()
    rc = lib.gelu_and_mul_sparse_typed(out.data_ptr(), x.data_ptr(), 8, 2048, 4096, W.Z95,
                                       ga.BF16, ga.VARIANT_AUTO, 0, 0)
    assert rc == ga.ERR_HOST
    rc = lib.silu_and_mul(out.data_ptr(), x.data_ptr(), 8, 1024, 0)
    assert rc == ga.ERR_HOST
    torch.cuda.synchronize()
