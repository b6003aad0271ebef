"""GPU parity of the widened rows against the fp64 oracle, through the C ABI:
silu_and_mul_bounded (device-side live-row count), dense gelu_and_mul and
squared_relu."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import SENTINEL, guarded_empty, guards_intact, require_gpu
from tests.parity import bits_of, check_silu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


# ------------------------------------------------------------ silu_and_mul_bounded
@pytest.mark.parametrize("n", [0, 1, 511, 512, 513, 1500, 2048, 5000, -3])
def test_bounded_silu_live_rows_only(ga, oracle, n):
    M, d = 2048, 768
    x = W.silu(M, d)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x))
    live = min(max(n, 0), M)
    out = torch.full((M, d), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    nr = torch.tensor([n], dtype=torch.int32, device="cuda")
    ga.silu_and_mul_bounded(x.cuda(), nr, out=out)
    torch.cuda.synchronize()
    if live:
        check_silu(out[:live], ref16[:live], f"bounded n={n}")
    assert (out[live:].view(torch.int16) == SENTINEL).all().item()


def test_bounded_silu_equals_unbounded_on_live_rows(ga):
    x = W.silu(4096).cuda()
    full = ga.silu_and_mul(x)
    part = ga.silu_and_mul_bounded(x, torch.tensor([3000], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(full[:3000].view(torch.int16), part[:3000].view(torch.int16))


def test_bounded_silu_one_graph_many_counts(ga, oracle):
    # the launch depends only on M: one capture serves every live count
    M, d = 16384, 768
    x = W.silu(M, d)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x))
    xd = x.cuda()
    out = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
    nr = torch.tensor([M], dtype=torch.int32, device="cuda")
    ga.silu_and_mul_bounded(xd, nr, out=out)          # first call outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ga.silu_and_mul_bounded(xd, nr, out=out)
    for n in (256, 8191, 1, M):
        out.view(torch.int16).fill_(SENTINEL)
        nr.fill_(n)
        g.replay()
        torch.cuda.synchronize()
        check_silu(out[:n], ref16[:n], f"graph n={n}")
        assert (out[n:].view(torch.int16) == SENTINEL).all().item()


def test_bounded_silu_ragged_layout_scalar_path(ga, oracle):
    M, d = 37, 33
    g = torch.Generator().manual_seed(4)
    x = torch.randn((M, 2 * d), generator=g).to(torch.bfloat16)
    _, ref16 = oracle.silu_and_mul(W.to_bits(x), d=d)
    out = torch.zeros((M, d), dtype=torch.bfloat16, device="cuda").view(torch.int16).fill_(SENTINEL)
    out = out.view(torch.bfloat16)
    ga.silu_and_mul_bounded(x.cuda(), torch.tensor([20], dtype=torch.int32, device="cuda"), out=out)
    torch.cuda.synchronize()
    check_silu(out[:20], ref16[:20], "bounded scalar")
    assert (out[20:].view(torch.int16) == SENTINEL).all().item()


# ------------------------------------------------------------ gelu_and_mul (dense)
@pytest.mark.parametrize("T,d,rs", [(4, 2048, None), (64, 8192, None), (2048, 16384, None),
                                    (9, 1000, 2048), (5, 33, 70), (3, 8, 24), (1, 1, 2)])
def test_dense_gelu_and_mul(ga, oracle, T, d, rs):
    inp = W.iid(T, d, seed=T * 13 + d, row_stride=rs)
    _, ref16 = oracle.gelu_and_mul(W.to_bits(inp.x), d=d)
    out = ga.gelu_and_mul(inp.x.cuda(), d=d)
    torch.cuda.synchronize()
    check_silu(out, ref16, f"gelu_and_mul T{T} d{d}")


def test_dense_gelu_and_mul_extremes(ga, oracle):
    vals = torch.tensor([0.0, -0.0, 0.5, -0.5, 3.0, -3.0, -5.5, -8.0, -10.0, -10.4, -11.0, -20.0,
                         12.0, 80.0, 1e-20, float("inf"), float("-inf"), float("nan")])
    d = vals.numel()
    x = torch.cat([vals, torch.linspace(-2, 2, d)]).reshape(1, 2 * d).repeat(4, 1)
    x = x.to(torch.bfloat16)
    _, ref16 = oracle.gelu_and_mul(W.to_bits(x), d=d)
    check_silu(ga.gelu_and_mul(x.cuda(), d=d), ref16, "gelu extremes")


def test_dense_gelu_vector_and_scalar_paths_agree(ga):
    T, d = 300, 1024
    x = W.iid(T, d, seed=1).x
    a = ga.gelu_and_mul(x.cuda())
    big = torch.zeros((T * 2 * d + 8,), dtype=torch.bfloat16, device="cuda")
    big[1:1 + T * 2 * d] = x.reshape(-1).cuda()
    b = ga.gelu_and_mul(big[1:1 + T * 2 * d].view(T, 2 * d))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------ squared_relu
@pytest.mark.parametrize("M,d", [(2048, 768), (16384, 768), (7, 33), (1, 1), (3, 4104)])
def test_squared_relu_exact(ga, oracle, M, d):
    g = torch.Generator().manual_seed(M + d)
    x = (3 * torch.randn((M, d), generator=g)).to(torch.bfloat16)
    _, ref16 = oracle.squared_relu_rows(W.to_bits(x))
    buf, out = guarded_empty((M, d))
    ga.squared_relu(x.cuda(), out=out)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert np.array_equal(bits_of(out), ref16)


def test_squared_relu_special_values(ga, oracle):
    x = torch.tensor([[0.0, -0.0, -1.0, 1.5, 1e20, 2e19, float("inf"), float("-inf"),
                       float("nan"), 1e-30, -1e-30, 3e38]], dtype=torch.bfloat16)
    _, ref16 = oracle.squared_relu_rows(W.to_bits(x))
    got = bits_of(ga.squared_relu(x.cuda()))
    nan = (ref16 & 0x7FFF) > 0x7F80
    assert np.array_equal((got & 0x7FFF) > 0x7F80, nan)
    # +0 and -0 compare equal
    same = (got == ref16) | (((got | ref16) & 0x7FFF) == 0)
    assert np.all(same | nan)


# ------------------------------------------------------------ 2^31-vector launches
def test_squared_relu_across_the_31_bit_index_boundary(ga, oracle):
    """Elementwise launches of fewer than 2^31 - 512 16-byte vectors index
    them in 32 bits, larger ones in 64 bits.  At d = 8 a row is one vector:
    2^31 - 4096 rows take the 32-bit kernel, 2^31 + 4096 rows the 64-bit one
    (64 GB of device memory in all).  Four windows of random rows, at the
    start, on both sides of row 2^31 - 4096 and at the end, are checked bit
    for bit against the oracle; the other rows are zero, and every output
    element is written exactly where it should be."""
    d, W_ = 8, 4096
    M_big, M_small = (1 << 31) + W_, (1 << 31) - W_
    free, _ = torch.cuda.mem_get_info()
    if free < 2 * M_big * d * 2 + (4 << 30):
        pytest.skip("needs about 68 GB of free device memory")
    x = out = None
    try:
        x = torch.zeros((M_big, d), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((M_big, d), dtype=torch.bfloat16, device="cuda")
        o16 = out.view(torch.int16)
        g = torch.Generator().manual_seed(31)
        starts = [0, M_small - W_, M_small, M_big - W_]
        refs = {}
        for s in starts:
            v = (3 * torch.randn((W_, d), generator=g)).to(torch.bfloat16)
            x[s:s + W_] = v.cuda()
            refs[s] = oracle.squared_relu_rows(W.to_bits(v))[1]

        def window(s):
            return bits_of(out[s:s + W_])

        def no_sentinel(lo, hi):
            step = 1 << 27   # rows per chunk: 2 GB of int16 compared at a time
            for a in range(lo, hi, step):
                if (o16[a:min(a + step, hi)] == SENTINEL).any().item():
                    return False
            return True

        # 32-bit indices: rows [0, M_small) written, the rest untouched
        o16.fill_(SENTINEL)
        ga.squared_relu(x[:M_small], out=out[:M_small])
        torch.cuda.synchronize()
        assert np.array_equal(window(0), refs[0])
        assert np.array_equal(window(M_small - W_), refs[M_small - W_])
        assert bool((o16[M_small:] == SENTINEL).all().item())
        assert no_sentinel(0, M_small)

        # 64-bit indices: every row written
        o16.fill_(SENTINEL)
        ga.squared_relu(x, out=out)
        torch.cuda.synchronize()
        for s in starts:
            assert np.array_equal(window(s), refs[s]), f"rows {s}..{s + W_}"
        assert no_sentinel(0, M_big)
        zero_rows = [W_, 1 << 20, (1 << 30) + 12345, M_small - 2 * W_ - 1]
        for r in zero_rows:
            assert int((o16[r] != 0).sum().item()) == 0, f"row {r}"
    finally:
        del x, out
        torch.cuda.empty_cache()
