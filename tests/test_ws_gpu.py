"""Dynamic rows (gelu_and_mul_sparse_ws): parity with the oracle, bitwise
equality with the round-robin path, the workspace left zeroed after every
call (also across a replayed graph and two streams), and its argument checks."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def _bits(t):
    return t.detach().cpu().view(torch.int16)


def _zeroed(ws) -> bool:
    return bool((ws == 0).all().item())


# (T, d): forced bulk-copy geometry, so rows are taken dynamically at any T:
# fewer rows than CTAs, ragged vector counts, widths up to the geometry's limit
# (more rows than CTAs for d >= 2048 at T >= 2433, 4096 at 1217, 8192 at 609,
# 32768 at 153)
FORCED = [(1, 2048), (5, 4096), (300, 4096), (2000, 1000), (5000, 2048), (3000, 4096),
          (700, 8192), (2500, 8192), (160, 32768), (3, 32768)]


@pytest.mark.parametrize("T,d", FORCED)
def test_dynamic_rows_match_oracle_and_static_path(ga, oracle, T, d):
    inp = W.sweep(T, d)
    x = inp.x.cuda()
    ws = ga.new_workspace()
    dyn = ga.gelu_and_mul_sparse(x, inp.z, variant=ga.VARIANT_TMA_ROWS, workspace=ws)
    stat = ga.gelu_and_mul_sparse(x, inp.z, variant=ga.VARIANT_TMA_ROWS)
    torch.cuda.synchronize()
    assert ga.gelu_and_mul_sparse_plan(x, variant=ga.VARIANT_TMA_ROWS)["dynamic_rows"] == 1
    assert _zeroed(ws)
    # one CTA computes each row either way: the bits agree
    assert torch.equal(_bits(dyn), _bits(stat))
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    check_gelu(dyn.cpu(), inp.x, d, res, f"dynamic T{T} d{d}")


# (T, d, geometry with a workspace, same geometry without one)
@pytest.mark.parametrize("T,d,kind,same", [(2048, 16384, "pipe_rows", True),
                                           (1024, 32768, "pipe_rows", True),
                                           (1100, 32768, "pipe_rows", True),
                                           (2048, 32768, "pipe_rows", False)])
def test_auto_geometry_with_workspace(ga, oracle, T, d, kind, same):
    inp = W.iid(T, d, seed=T + 7 * d)
    x = inp.x.cuda()
    plan = ga.gelu_and_mul_sparse_plan(x, workspace=True)
    assert plan["variant"] == kind and plan["dynamic_rows"] == 1
    assert (ga.gelu_and_mul_sparse_plan(x) == plan) == same
    ws = ga.new_workspace()
    out = ga.gelu_and_mul_sparse(x, inp.z, workspace=ws)
    torch.cuda.synchronize()
    assert _zeroed(ws)
    if same:   # the same geometry computes every row in the same order
        assert torch.equal(_bits(out), _bits(ga.gelu_and_mul_sparse(x, inp.z)))
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    check_gelu(out.cpu(), inp.x, d, res, f"auto+ws T{T} d{d}")


def test_workspace_ignored_by_other_geometries(ga):
    inp = W.iid(64, 4096, seed=3)
    x = inp.x.cuda()
    assert ga.gelu_and_mul_sparse_plan(x)["dynamic_rows"] == 0
    ws = ga.new_workspace()
    a = ga.gelu_and_mul_sparse(x, inp.z, workspace=ws)
    b = ga.gelu_and_mul_sparse(x, inp.z)
    torch.cuda.synchronize()
    assert torch.equal(_bits(a), _bits(b)) and _zeroed(ws)


def test_one_workspace_across_a_replayed_graph(ga):
    # 12 launches of two shapes share one workspace inside a graph replayed
    # three times; each launch must find it zeroed by the one before
    shapes = [(3000, 4096), (5000, 2048)] * 6
    xs = [W.iid(T, d, seed=50 + i).x.cuda() for i, (T, d) in enumerate(shapes)]
    outs = [torch.empty((T, d), dtype=torch.bfloat16, device="cuda") for T, d in shapes]
    refs = [ga.gelu_and_mul_sparse(x, W.Z95, variant=ga.VARIANT_TMA_ROWS) for x in xs]
    ws = ga.new_workspace()
    for x, o in zip(xs, outs):   # first calls (shared-memory set-up) before capture
        ga.gelu_and_mul_sparse(x, W.Z95, out=o, variant=ga.VARIANT_TMA_ROWS, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for x, o in zip(xs, outs):
            ga.gelu_and_mul_sparse(x, W.Z95, out=o, variant=ga.VARIANT_TMA_ROWS, workspace=ws)
    for _ in range(3):
        for o in outs:
            o.view(torch.int16).fill_(0x7FA1)
        g.replay()
        torch.cuda.synchronize()
        assert _zeroed(ws)
        for o, r in zip(outs, refs):
            assert torch.equal(_bits(o), _bits(r))


def test_two_streams_two_workspaces(ga):
    xa = W.iid(1500, 8192, seed=11).x.cuda()
    xb = W.iid(900, 16384, seed=12).x.cuda()
    ra = ga.gelu_and_mul_sparse(xa, W.Z95, variant=ga.VARIANT_TMA_ROWS)
    rb = ga.gelu_and_mul_sparse(xb, W.Z95, variant=ga.VARIANT_TMA_ROWS)
    torch.cuda.synchronize()
    wa, wb = ga.new_workspace(), ga.new_workspace()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    oa, ob = [], []
    for _ in range(4):
        oa.append(ga.gelu_and_mul_sparse(xa, W.Z95, variant=ga.VARIANT_TMA_ROWS,
                                         workspace=wa, stream=sa))
        ob.append(ga.gelu_and_mul_sparse(xb, W.Z95, variant=ga.VARIANT_TMA_ROWS,
                                         workspace=wb, stream=sb))
    torch.cuda.synchronize()
    assert _zeroed(wa) and _zeroed(wb)
    for o in oa:
        assert torch.equal(_bits(o), _bits(ra))
    for o in ob:
        assert torch.equal(_bits(o), _bits(rb))


def test_workspace_argument_checks(ga):
    lib = ga.load_library()
    x = W.iid(300, 4096, seed=1).x.cuda()
    out = torch.empty((300, 4096), dtype=torch.bfloat16, device="cuda")
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")

    def call(ws_ptr):
        return lib.gelu_and_mul_sparse_ws(out.data_ptr(), x.data_ptr(), 300, 4096, 8192, W.Z95,
                                          ga.BF16, ga.VARIANT_TMA_ROWS, 0, ws_ptr, 0)

    assert call(None) == ga.ERR_NULL
    assert call(buf.data_ptr() + 4) == ga.ERR_ALIGN
    assert call(out.data_ptr() + 64) == ga.ERR_OVERLAP
    pinned = torch.zeros(16, dtype=torch.uint8).pin_memory()
    assert call(pinned.data_ptr()) == ga.ERR_HOST
    pageable = np.zeros(4, dtype=np.uint64)
    assert call(pageable.ctypes.data) == ga.ERR_HOST
    torch.cuda.synchronize()
    assert (buf == 0).all().item()


def test_workspace_with_host_buffers_is_ignored(ga, oracle):
    # page-locked host rows never take the bulk-copy geometry, so the
    # workspace is not used and stays zeroed
    inp = W.iid(2048, 16384, seed=21)
    x = inp.x.pin_memory()
    ws = ga.new_workspace()
    assert ga.gelu_and_mul_sparse_plan(x)["dynamic_rows"] == 0
    out = ga.gelu_and_mul_sparse(x, inp.z, workspace=ws)
    torch.cuda.synchronize()
    assert not out.is_cuda and _zeroed(ws)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=16384, z=inp.z)
    check_gelu(out, inp.x, 16384, res, "host rows with a workspace")
