"""Failure handling of the bounded waits, on the GPU without a fault: every
CTA of a TMA-rows or pipe-rows launch withholds one bulk copy, so its wait
runs out after a short limit.  The kernel must record the status bit, drain
its own copies and return; the context must stay usable and later calls
correct."""
import ctypes

import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def test_wait_runs_out_and_is_reported(ga, oracle):
    assert ga.device_status() == 0
    inp = W.iid(400, 4096, seed=11)
    x = inp.x.cuda()
    out = torch.zeros((400, 4096), dtype=torch.bfloat16, device="cuda")
    lib = ga.load_library()
    rc = lib.gated_act_selftest_wait_timeout(out.data_ptr(), x.data_ptr(), 400, 4096,
                                             20_000_000, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()              # the launch ends: every wait was bounded
    assert ga.device_status() == 1        # bit 0: a wait gave up
    assert ga.device_status() == 0        # reading clears it
    # the context is usable and the same kernel is correct without the fault
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=4096, z=inp.z)
    good = ga.gelu_and_mul_sparse(x, inp.z, variant=ga.VARIANT_TMA_ROWS)
    torch.cuda.synchronize()
    check_gelu(good.cpu(), inp.x, 4096, res, "after timeout")
    assert ga.device_status() == 0


def test_selftest_rejects_unbounded_limits(ga):
    lib = ga.load_library()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((4, 32), dtype=torch.bfloat16, device="cuda")
    assert lib.gated_act_selftest_wait_timeout(o.data_ptr(), x.data_ptr(), 4, 32, 0, None) == ga.ERR_SIZE
    assert lib.gated_act_selftest_wait_timeout(o.data_ptr(), x.data_ptr(), 4, 32, 2_000_000_000,
                                               None) == ga.ERR_SIZE


def test_wait_runs_out_with_dynamic_rows(ga, oracle):
    # rows taken from a workspace: every CTA gives up on its first row's up
    # half, still counts itself out, and the last one resets the workspace
    assert ga.device_status() == 0
    inp = W.iid(2000, 4096, seed=12)      # more rows than CTAs: tickets are taken
    x = inp.x.cuda()
    out = torch.zeros((2000, 4096), dtype=torch.bfloat16, device="cuda")
    ws = ga.new_workspace()
    lib = ga.load_library()
    rc = lib.gated_act_selftest_wait_timeout_ws(out.data_ptr(), x.data_ptr(), 2000, 4096,
                                                20_000_000, ws.data_ptr(),
                                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert ga.device_status() == 1
    assert int(ws.count_nonzero().item()) == 0
    good = ga.gelu_and_mul_sparse(x, inp.z, variant=ga.VARIANT_TMA_ROWS, workspace=ws)
    torch.cuda.synchronize()
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=4096, z=inp.z)
    check_gelu(good.cpu(), inp.x, 4096, res, "dynamic rows after timeout")
    assert int(ws.count_nonzero().item()) == 0 and ga.device_status() == 0
    assert lib.gated_act_selftest_wait_timeout_ws(out.data_ptr(), x.data_ptr(), 4, 4096,
                                                  20_000_000, None, None) == ga.ERR_NULL


@pytest.mark.parametrize("dynamic", [False, True])
@pytest.mark.parametrize("T,d", [(400, 4096), (2000, 8192), (300, 32768)])
def test_wait_runs_out_in_pipe_rows(ga, oracle, T, d, dynamic):
    # consumers give up on their first row's up half and stop together; the
    # producer lane stops issuing, drains its copies and (dynamic rows) leaves
    # the workspace zeroed
    assert ga.device_status() == 0
    inp = W.iid(T, d, seed=T + d)
    x = inp.x.cuda()
    out = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    ws = ga.new_workspace() if dynamic else None
    lib = ga.load_library()
    rc = lib.gated_act_selftest_wait_timeout_ex(out.data_ptr(), x.data_ptr(), T, d, 20_000_000,
                                                ga.VARIANT_PIPE_ROWS,
                                                ws.data_ptr() if dynamic else None,
                                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert ga.device_status() == 1
    assert ga.device_status() == 0
    if dynamic:
        assert int(ws.count_nonzero().item()) == 0
    good = ga.gelu_and_mul_sparse(x, inp.z, variant=ga.VARIANT_PIPE_ROWS, workspace=ws)
    torch.cuda.synchronize()
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    check_gelu(good.cpu(), inp.x, d, res, "pipe rows after timeout")
    assert ga.device_status() == 0
    if dynamic:
        assert int(ws.count_nonzero().item()) == 0


def test_selftest_ex_argument_checks(ga):
    lib = ga.load_library()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((4, 32), dtype=torch.bfloat16, device="cuda")
    for bad_variant in (ga.VARIANT_AUTO, ga.VARIANT_CTA_ROW, 9):
        assert lib.gated_act_selftest_wait_timeout_ex(o.data_ptr(), x.data_ptr(), 4, 32, 1000,
                                                      bad_variant, None, None) == ga.ERR_VARIANT
    assert lib.gated_act_selftest_wait_timeout_ex(o.data_ptr(), x.data_ptr(), 4, 32, 0,
                                                  ga.VARIANT_PIPE_ROWS, None, None) == ga.ERR_SIZE
