"""GPU parity of gelu_and_mul_sparse against the fp64 oracle, through the C ABI.

Every config of the workload set (tiny, decode, prefill, the T x d x z sweep
with constant rows), every launch geometry, and the edge cases: empty, d=1,
ragged widths, strided and misaligned rows, NaN, maximum on-chip widths,
guard-band canaries and CUDA-graph capture.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import guarded_empty, guards_intact, require_gpu
from tests.parity import bits_of, check_gelu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def run(ga, x_cpu, d, z, **kw):
    x = x_cpu.to("cuda")
    out = ga.gelu_and_mul_sparse(x, z, d=d, **kw)
    torch.cuda.synchronize()
    return out.cpu()


def oracle_of(oracle, x_cpu, d, z):
    return oracle.gelu_and_mul_sparse(W.to_bits(x_cpu.contiguous()), d=d, z=z)


GEOMETRIES = [(0, 0), (1, 0), (2, 1), (2, 2), (2, 4), (2, 8), (3, 0), (4, 0), (5, 0), (5, 1),
              (6, 2), (6, 4), (6, 8)]


@pytest.mark.parametrize("variant,cluster", GEOMETRIES)
def test_tiny_every_geometry(ga, oracle, variant, cluster):
    inp = W.tiny()
    res = oracle_of(oracle, inp.x, inp.d, inp.z)
    out = run(ga, inp.x, inp.d, inp.z, variant=variant, cluster=cluster)
    check_gelu(out, inp.x, inp.d, res, f"tiny v{variant} c{cluster}")


@pytest.mark.parametrize("T", W.DECODE_T)
def test_decode(ga, oracle, T):
    inp = W.decode(T)
    res = oracle_of(oracle, inp.x, inp.d, inp.z)
    out = run(ga, inp.x, inp.d, inp.z)
    check_gelu(out, inp.x, inp.d, res, inp.name)


@pytest.mark.parametrize("variant,cluster", [(2, 1), (2, 2), (2, 4), (2, 8), (6, 2), (6, 4),
                                             (6, 8)])
def test_decode_forced_clusters(ga, oracle, variant, cluster):
    # the decode workload (outliers in the gate) in clusters and in split rows
    inp = W.decode(16)
    res = oracle_of(oracle, inp.x, inp.d, inp.z)
    out = run(ga, inp.x, inp.d, inp.z, variant=variant, cluster=cluster)
    check_gelu(out, inp.x, inp.d, res, f"decode16 v{variant} c{cluster}")


# few wide rows that the plan spreads over several CTAs: split rows
# (independent CTAs, each with the whole row's statistics) while they fit one
# wave -- at any row count above d = 8192 up to 20480, from 9 rows at d =
# 8192 (8 or 4 CTAs per row) and wider -- and 8-CTA clusters for up to 8 rows
# wider than 20480 (rows = T random rows + 3 constant rows)
@pytest.mark.parametrize("rows,d,variant,cluster", [
    (4, 16384, "split_rows", 8), (9, 16384, "split_rows", 8), (16, 16384, "split_rows", 8),
    (24, 16384, "split_rows", 4), (33, 16384, "split_rows", 4), (64, 16384, "split_rows", 2),
    (80, 16384, "cta_row", 1), (16, 20480, "split_rows", 8), (32, 24576, "split_rows", 4),
    (48, 24576, "split_rows", 2), (70, 32768, "split_rows", 2), (4, 9216, "split_rows", 8),
    (16, 11008, "split_rows", 8), (24, 14336, "split_rows", 4), (60, 12288, "split_rows", 2),
    (20, 8192, "split_rows", 4), (40, 8192, "cta_row", 1), (4, 32768, "cta_row", 8),
    (8, 24576, "cta_row", 8), (12, 32768, "split_rows", 8)])
def test_wide_few_rows_spread_over_ctas(ga, oracle, rows, d, variant, cluster):
    inp = W.sweep(rows - 3, d, z=W.Z95, const_rows=True)
    assert inp.x.shape[0] == rows
    plan = ga.gelu_and_mul_sparse_plan(inp.x.cuda(), d=inp.d)
    assert plan["variant"] == variant and plan["cluster"] == cluster, plan
    res = oracle_of(oracle, inp.x, inp.d, inp.z)
    out = run(ga, inp.x, inp.d, inp.z)
    check_gelu(out, inp.x, inp.d, res, f"{inp.name} {variant} c{cluster}")
    assert torch.count_nonzero(out[-3:].float()).item() == 0


# split rows forced: every CTA count, ragged widths (the last slice short or
# empty), fp16 and fp32 rows, strided rows with NaN in the padding
@pytest.mark.parametrize("T,d,c,dtype,pad", [
    (5, 16384, 2, torch.bfloat16, 0), (7, 16384, 4, torch.bfloat16, 0),
    (3, 16384, 8, torch.bfloat16, 0), (6, 32768, 8, torch.bfloat16, 0),
    (4, 16392, 8, torch.bfloat16, 0), (9, 1000, 8, torch.bfloat16, 0),
    (11, 8, 2, torch.bfloat16, 0), (6, 16384, 4, torch.float16, 0),
    (6, 8192, 8, torch.float32, 0), (5, 12296, 4, torch.bfloat16, 24)])
def test_split_rows_forced(ga, oracle, T, d, c, dtype, pad):
    inp = W.iid(T, d, seed=T * 7 + d + c, row_stride=2 * d + pad, dtype=dtype)
    x = inp.x.clone()
    if pad:
        x[:, 2 * d:] = float("nan")
    out = ga.gelu_and_mul_sparse(x.cuda(), inp.z, d=d, variant=ga.VARIANT_SPLIT_ROWS, cluster=c)
    torch.cuda.synchronize()
    if dtype == torch.bfloat16:
        res = oracle.gelu_and_mul_sparse(W.to_bits(x), d=d, z=inp.z)
    else:
        res = oracle.gelu_and_mul_sparse_typed(x.contiguous().numpy(), d=d, z=inp.z)
    check_gelu(out.cpu(), x, d, res, f"split T{T} d{d} c{c} {dtype}")


# many rows of d = 28672 without a workspace: tma rows (round-robin rows)
def test_wide_rows_without_workspace_take_tma_rows(ga, oracle):
    inp = W.sweep(1216, 28672, z=W.Z95, const_rows=True)
    plan = ga.gelu_and_mul_sparse_plan(inp.x.cuda(), d=inp.d)
    assert plan["variant"] == "tma_rows", plan
    res = oracle_of(oracle, inp.x, inp.d, inp.z)
    check_gelu(run(ga, inp.x, inp.d, inp.z), inp.x, inp.d, res, f"{inp.name} tma rows")


def test_prefill_full(ga, oracle):
    inp = W.prefill()
    res = oracle_of(oracle, inp.x, inp.d, inp.z)
    out = run(ga, inp.x, inp.d, inp.z)
    stats = check_gelu(out, inp.x, inp.d, res, "prefill")
    assert abs(stats["zero_fraction"] - 0.95) < 0.003


@pytest.mark.parametrize("z", W.SWEEP_Z)
@pytest.mark.parametrize("d", W.SWEEP_D)
@pytest.mark.parametrize("T", W.SWEEP_T)
def test_sweep(ga, oracle, T, d, z):
    inp = W.sweep(T, d, z=z, const_rows=True)
    res = oracle_of(oracle, inp.x, inp.d, z)
    out = run(ga, inp.x, inp.d, z)
    check_gelu(out, inp.x, inp.d, res, f"{inp.name} z={z}")
    # the three constant-gate rows: std == 0, exact zeros
    tail = out[-len(W.CONST_GATES):].to(torch.float32)
    assert torch.count_nonzero(tail).item() == 0


@pytest.mark.parametrize("z", W.SWEEP_Z)
@pytest.mark.parametrize("d", W.SWEEP_D)
@pytest.mark.parametrize("T", W.SWEEP_T)
def test_sweep_in_the_bench_configuration(ga, oracle, T, d, z):
    """The timed launches exactly: T rows (no appended rows), the bench's input
    (seed 7919 T + d), a workspace, the library's own geometry."""
    x = W.iid(T, d, seed=W.sweep_seed(T, d), z=z).x
    res = oracle_of(oracle, x, d, z)
    ws = ga.new_workspace()
    xd = x.to("cuda")
    plan = ga.gelu_and_mul_sparse_plan(xd, d=d, workspace=True)
    out = ga.gelu_and_mul_sparse(xd, z, d=d, workspace=ws)
    torch.cuda.synchronize()
    check_gelu(out.cpu(), x, d, res, f"bench T{T} d{d} z={z} ({plan['variant']})")
    assert int(ws.count_nonzero().item()) == 0


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("T,d", [(8, 8192), (64, 16384), (3, 32768)])
def test_sweep_shapes_every_cluster(ga, oracle, T, d, cluster):
    inp = W.sweep(T, d, const_rows=True)
    res = oracle_of(oracle, inp.x, d, inp.z)
    if (d // 8 + cluster - 1) // cluster > 4096:
        pytest.skip("slice does not fit one CTA")
    out = run(ga, inp.x, d, inp.z, variant=2, cluster=cluster)
    check_gelu(out, inp.x, d, res, f"{inp.name} c{cluster}")


@pytest.mark.parametrize("T,d", [(2048, 2048), (1024, 4096), (512, 8192), (300, 16384),
                                 (257, 32768), (5, 16384), (1, 2048), (1000, 1024), (777, 2056),
                                 (333, 8200)])
def test_tma_rows_forced(ga, oracle, T, d):
    inp = W.iid(T, d, seed=T * 7 + d)
    res = oracle_of(oracle, inp.x, d, inp.z)
    out = run(ga, inp.x, d, inp.z, variant=4)
    check_gelu(out, inp.x, d, res, f"tma T{T} d{d}")
    assert ga.device_status() == 0


def test_tma_rows_strided_and_constant_rows(ga, oracle):
    inp = W.sweep(1024, 8192, const_rows=True)
    res = oracle_of(oracle, inp.x, 8192, inp.z)
    out = run(ga, inp.x, 8192, inp.z, variant=4)
    check_gelu(out, inp.x, 8192, res, "tma sweep rows")
    assert torch.count_nonzero(out[-3:].float()).item() == 0
    inp = W.iid(700, 4096, seed=3, row_stride=8192 + 64)
    res = oracle_of(oracle, inp.x, 4096, inp.z)
    out = run(ga, inp.x, 4096, inp.z, variant=4)
    check_gelu(out, inp.x, 4096, res, "tma strided")
    assert ga.device_status() == 0


def test_same_geometry_is_bitwise_deterministic(ga):
    inp = W.sweep(64, 8192, const_rows=False)
    x = inp.x.cuda()
    a = ga.gelu_and_mul_sparse(x, inp.z)
    b = ga.gelu_and_mul_sparse(x, inp.z)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("T,d", [(1, 1), (5, 1), (3, 2), (4, 7), (9, 8), (5, 16), (3, 24), (7, 31),
                                 (4, 33), (6, 128), (2, 255), (3, 2056), (2, 4104), (2, 16392),
                                 (37, 1000), (2, 32776)])
def test_ragged_widths(ga, oracle, T, d):
    inp = W.iid(T, d, seed=T * 1009 + d)
    res = oracle_of(oracle, inp.x, d, inp.z)
    out = run(ga, inp.x, d, inp.z)
    check_gelu(out, inp.x, d, res, f"T{T} d{d}")
    if d == 1:
        assert torch.count_nonzero(out.float()).item() == 0


@pytest.mark.parametrize("d,extra", [(64, 8), (2048, 16), (8192, 8), (1000, 24), (64, 3), (2048, 1)])
def test_strided_rows_never_read_padding(ga, oracle, d, extra):
    # padding columns hold NaN: any read of them would poison the row
    inp = W.iid(11, d, seed=d + extra, row_stride=2 * d + extra)
    res = oracle_of(oracle, inp.x, d, inp.z)
    x = inp.x.cuda()
    out = ga.gelu_and_mul_sparse(x, inp.z, d=d)
    torch.cuda.synchronize()
    check_gelu(out.cpu(), inp.x, d, res, f"strided d{d}+{extra}")


@pytest.mark.parametrize("offset", [1, 2, 3, 4])
def test_misaligned_input_pointer(ga, oracle, offset):
    d, T = 2048, 6
    inp = W.iid(T, d, seed=offset)
    big = torch.zeros((T * 2 * d + 8,), dtype=torch.bfloat16)
    big[offset:offset + T * 2 * d] = inp.x.reshape(-1)
    gbig = big.cuda()
    x = gbig[offset:offset + T * 2 * d].view(T, 2 * d)
    out = ga.gelu_and_mul_sparse(x, inp.z)
    torch.cuda.synchronize()
    res = oracle_of(oracle, inp.x, d, inp.z)
    check_gelu(out.cpu(), inp.x, d, res, f"offset {offset}")


def test_guard_bands_untouched(ga, oracle):
    for T, d, v in ((4, 2048, 0), (64, 8192, 0), (5, 31, 0), (3, 32768, 0), (2048, 4096, 0),
                    (2048, 4096, 4), (600, 32768, 4), (7, 2048, 4), (2048, 4096, 5),
                    (600, 32768, 5), (7, 2048, 5)):
        inp = W.iid(T, d, seed=T + d)
        buf, out = guarded_empty((T, d))
        ga.gelu_and_mul_sparse(inp.x.cuda(), inp.z, out=out, variant=v)
        torch.cuda.synchronize()
        assert guards_intact(buf), (T, d, v)
        check_gelu(out.cpu(), inp.x, d, oracle_of(oracle, inp.x, d, inp.z), f"guard T{T} d{d} v{v}")


# the plan's choice at d = 2048, and split rows (each CTA of a row reads the
# NaN for its statistics, so every slice of the row is NaN)
@pytest.mark.parametrize("d,kw", [(2048, {}), (16384, {"variant": 6, "cluster": 8}),
                                  (32768, {"variant": 6, "cluster": 2})])
def test_nan_poisons_only_its_row(ga, oracle, d, kw):
    inp = W.iid(6, d, seed=17)
    x = inp.x.clone()
    x[2, d - 100] = float("nan")        # in the gate (the last slice): row 2 all NaN
    x[4, d + 7] = float("nan")          # in up: one element
    out = run(ga, x, d, inp.z, **kw)
    res = oracle_of(oracle, x, d, inp.z)
    check_gelu(out, x, d, res, f"nan d{d}")
    o = out.float()
    assert torch.isnan(o[2]).all()
    assert torch.isnan(o[4]).sum().item() <= 1
    assert not torch.isnan(o[[0, 1, 3, 5]]).any()


def test_zero_rows(ga):
    x = torch.empty((0, 4096), dtype=torch.bfloat16, device="cuda")
    out = ga.gelu_and_mul_sparse(x, W.Z95)
    assert out.shape == (0, 2048)


@pytest.mark.parametrize("T,d", [(3, 131072), (2, 262144), (2, 262152), (2, 1 << 20)])
def test_widest_rows(ga, oracle, T, d):
    inp = W.iid(T, d, seed=d)
    res = oracle_of(oracle, inp.x, d, inp.z)
    out = run(ga, inp.x, d, inp.z)
    check_gelu(out, inp.x, d, res, f"wide d{d}")


def test_many_short_rows(ga, oracle):
    inp = W.iid(100003, 8, seed=5)
    res = oracle_of(oracle, inp.x, 8, inp.z)
    out = run(ga, inp.x, 8, inp.z)
    check_gelu(out, inp.x, 8, res, "many rows")


def test_device_status_clear_after_the_suite(ga):
    assert ga.device_status() == 0


def test_side_stream_and_graph_capture(ga):
    inps = [W.sweep(T, d, const_rows=False) for T, d in ((8, 8192), (256, 4096), (2048, 2048),
                                                          (2048, 16384))]
    xs = [i.x.cuda() for i in inps]
    eager = [ga.gelu_and_mul_sparse(x, W.Z95) for x in xs]
    outs = [torch.empty_like(e) for e in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for x, o in zip(xs, outs):
            ga.gelu_and_mul_sparse(x, W.Z95, out=o)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for e, o in zip(eager, outs):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16))
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for x, o in zip(xs, outs):
            ga.gelu_and_mul_sparse(x, W.Z95, out=o)
    g.replay()
    torch.cuda.synchronize()
    for e, o in zip(eager, outs):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16))


# rows past 4 GB of input: every row offset needs 64-bit arithmetic
@pytest.mark.parametrize("T,d,workspace,kind", [
    (70000, 16384, False, "pipe_rows"),      # 4.6 GB of input
    (70000, 16384, True, "pipe_rows"),
    (36001, 32768, False, "tma_rows"),       # 4.7 GB
    (36001, 32768, True, "pipe_rows"),
    (140000, 8192, False, "cta_row"),        # 4.6 GB
])
def test_rows_past_4gb(ga, oracle, T, d, workspace, kind):
    """Seven random rows tiled over T rows (T a multiple of 7) on the device:
    the seven are checked against the oracle, and every other row must equal
    its source row bit for bit (each row is computed independently by the
    same code)."""
    assert T % 7 == 0
    need = T * 3 * d * 2 + (2 << 30)
    if torch.cuda.mem_get_info()[0] < need:
        pytest.skip("not enough free device memory")
    src = W.iid(7, d, seed=d + 7)
    res = oracle_of(oracle, src.x, d, src.z)
    ws = ga.new_workspace() if workspace else None
    x = out = None
    try:
        x = src.x.to("cuda").repeat(T // 7, 1)
        assert x.numel() * 2 > (1 << 32)
        assert ga.gelu_and_mul_sparse_plan(x, d=d, workspace=workspace)["variant"] == kind
        out = ga.gelu_and_mul_sparse(x, src.z, d=d, workspace=ws)
        torch.cuda.synchronize()
        check_gelu(out[:7].cpu(), src.x, d, res, f"{T}x{d} rows 0..6")
        o16 = out.view(torch.int16).view(T // 7, 7, d)
        same = (o16 == o16[0]).view(T // 7, -1).all(dim=1)
        assert bool(same.all().item()), f"first differing block {int((~same).nonzero()[0])}"
        if ws is not None:
            assert int(ws.count_nonzero().item()) == 0
    finally:
        del x, out
        torch.cuda.empty_cache()
