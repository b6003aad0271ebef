"""The producer/consumer geometry (gelu_pipe_rows): parity with the oracle at
every CTAs-per-SM setting it supports, round-robin and dynamic rows (bitwise
equal to each other, the latter with its last rows split in half jobs at
d = 32768), ragged widths, guard bands, the workspace left zeroed, and its
give-up path without a fault."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import guarded_empty, guards_intact, require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def _bits(t):
    return t.detach().cpu().view(torch.int16)


# (T, d, CTAs per SM; 0 = the library's choice): fewer rows than CTAs, a
# handful per CTA, many per CTA; widths that fill every consumer vector, and
# ragged ones (d = 1000: 125 vectors; d = 12296: 1537; d = 32760: 4095)
CASES = [(1, 2048, 0), (7, 4096, 4), (300, 4096, 4), (2000, 1000, 0), (5000, 2048, 4),
         (700, 8192, 2), (2500, 8192, 4), (1300, 8192, 1), (333, 12296, 0), (640, 16384, 2),
         (2048, 16384, 1), (160, 32768, 1), (3, 32768, 0), (1000, 32768, 1),
         # widths between the powers of two, and an odd vector count
         (300, 20480, 0), (600, 24576, 0), (200, 32760, 0), (257, 16392, 0),
         # dynamic rows with the last rows split in half jobs: just above the
         # threshold (3 rows per CTA), and more rows per CTA
         (460, 32768, 0), (1500, 32768, 0)]


@pytest.mark.parametrize("T,d,cps", CASES)
def test_pipe_rows_match_oracle_static_and_dynamic(ga, oracle, T, d, cps):
    inp = W.sweep(T, d)
    x = inp.x.cuda()
    plan = ga.gelu_and_mul_sparse_plan(x, variant=ga.VARIANT_PIPE_ROWS, cluster=cps)
    assert plan["variant"] == "pipe_rows"
    if cps:
        assert plan["ctas_per_sm"] == cps
    rows = x.shape[0]
    buf_s, stat = guarded_empty((rows, d))
    buf_d, dyn = guarded_empty((rows, d))
    ws = ga.new_workspace()
    ga.gelu_and_mul_sparse(x, inp.z, out=stat, variant=ga.VARIANT_PIPE_ROWS, cluster=cps)
    ga.gelu_and_mul_sparse(x, inp.z, out=dyn, variant=ga.VARIANT_PIPE_ROWS, cluster=cps,
                           workspace=ws)
    torch.cuda.synchronize()
    assert guards_intact(buf_s) and guards_intact(buf_d)
    assert bool((ws == 0).all().item()), "workspace not left zeroed"
    assert ga.device_status() == 0
    # whole rows or half jobs: the same statistics and arithmetic, so the same bits
    assert torch.equal(_bits(dyn), _bits(stat)), "dynamic rows differ from round-robin rows"
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    check_gelu(stat.cpu(), inp.x, d, res, f"pipe T{T} d{d} cps{cps}")


def test_pipe_rows_strided_rows_with_nan_padding(ga, oracle):
    # row_stride > 2d with NaN in the padding: a stray read would poison rows
    T, d = 900, 4096
    inp = W.iid(T, d, seed=11, row_stride=2 * d + 64)
    x = inp.x.cuda()
    out = ga.gelu_and_mul_sparse(x, inp.z, d=d, variant=ga.VARIANT_PIPE_ROWS)
    torch.cuda.synchronize()
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    check_gelu(out.cpu(), inp.x, d, res, "pipe strided")


def test_pipe_rows_repeated_in_a_graph_with_one_workspace(ga):
    T, d = 3000, 8192
    xs = [W.iid(T, d, seed=40 + i).x.cuda() for i in range(3)]
    refs = [ga.gelu_and_mul_sparse(x, W.Z95, variant=ga.VARIANT_PIPE_ROWS) for x in xs]
    outs = [torch.empty(T, d, dtype=torch.bfloat16, device="cuda") for _ in xs]
    ws = ga.new_workspace()
    for x, o in zip(xs, outs):   # first launches outside capture (shared-memory opt-in)
        ga.gelu_and_mul_sparse(x, W.Z95, out=o, variant=ga.VARIANT_PIPE_ROWS, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(2):
            for x, o in zip(xs, outs):
                ga.gelu_and_mul_sparse(x, W.Z95, out=o, variant=ga.VARIANT_PIPE_ROWS,
                                       workspace=ws)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert bool((ws == 0).all().item())
    for o, r in zip(outs, refs):
        assert torch.equal(_bits(o), _bits(r))
