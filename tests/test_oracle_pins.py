"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each pin is something the definitions or the mathematics fix -- IEEE bf16
encodings, library routines (torch / numpy / math.erf), closed forms, exact
special cases, brute force over tiny integer rows, invariances, and the
sparsity a Gaussian threshold must give -- chosen so that a plausible slip in
the oracle (a dropped term, a sign, sample instead of population variance,
swapped gate/up halves, a double rounding) fails at least one of them.

Definition pinned: vLLM PR "[Performance] Add Triton kernel for Gemma3n sparse
GELU", section "Purpose" (the fused stages: row statistics, a threshold from
them, tanh GELU, the product with the up half), read as
    out = gelu_tanh(relu(gate - (mean + std * z))) * up,  std = population std;
and Megatron-LM PR "Size MoE activation kernel grid to the row count",
section "What changed and why" (out = silu(gate) * up).
"""
import math
import statistics

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as W

Z95 = W.Z95


# ---------------------------------------------------------------- constants
def test_z_is_normal_quantile_of_target_sparsity():
    # Phi(z) = 0.5 erfc(-z / sqrt 2) must be the target sparsity 0.95
    assert abs(0.5 * math.erfc(-Z95 / math.sqrt(2.0)) - 0.95) < 1e-15
    assert abs(statistics.NormalDist().inv_cdf(0.95) - Z95) < 1e-14


# ---------------------------------------------------------------- bf16 codec
@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x3FC0, 1.5), (0x0000, 0.0),
    (0x0001, 2.0 ** -133), (0x0080, 2.0 ** -126), (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127),
    (0x7F80, math.inf), (0xFF80, -math.inf),
])
def test_bf16_decode_ieee_fields(oracle, bits, value):
    assert oracle.bf16_to_double(bits) == value


def test_bf16_decode_matches_torch_for_all_patterns(oracle):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = W.from_bits(bits).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_encode_matches_torch_on_binary32_values(oracle):
    # For values that are exactly binary32 there is no double rounding, so
    # torch's float32 -> bf16 cast (round to nearest even) is an independent
    # reference.  Includes subnormals, ties and values near overflow.
    rng = np.random.default_rng(5)
    w = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = w.view(np.float32)
    f = f[np.isfinite(f)]
    extra = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3 * 2 ** -134,
                      (2 - 2 ** -8) * 2 ** 127, (2 - 2 ** -9) * 2 ** 127], dtype=np.float32)
    f = np.concatenate([f, extra])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_rounds_once_from_double(oracle):
    # 1 + 2^-8 + 2^-40 lies just above the tie between 1 and 1 + 2^-7, so it
    # rounds up.  Going through binary32 first would land on the tie and round
    # to even (1.0): a double rounding.
    assert oracle.double_to_bf16(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.double_to_bf16(1 + 2 ** -8) == 0x3F80          # tie -> even
    assert oracle.double_to_bf16(1 + 3 * 2 ** -8) == 0x3F82      # tie -> even
    assert oracle.double_to_bf16(-0.0) == 0x8000
    assert oracle.double_to_bf16(1e300) == 0x7F80
    assert oracle.double_to_bf16(float("nan")) & 0x7FC0 == 0x7FC0


# ---------------------------------------------------------------- GELU (tanh)
def test_gelu_tanh_matches_torch_library(oracle):
    xs = np.concatenate([np.linspace(-10, 10, 4001), [0.0, 0.5, 1.0, 2.0, 3.0, 1e-8, 40.0]])
    ref = F.gelu(torch.tensor(xs, dtype=torch.float64), approximate="tanh").numpy()
    got = np.array([oracle.gelu_tanh(x) for x in xs])
    # torch evaluates 1 + tanh(y), which cancels for y << 0: compare absolutely
    # there, relatively where torch keeps its digits (x >= -2); the far-negative
    # tail is pinned against a 400-digit evaluation below.
    assert np.all(np.abs(got - ref) <= 1e-15)
    keep = xs >= -2.0
    assert np.allclose(got[keep], ref[keep], rtol=2e-14, atol=1e-300)


def test_gelu_tanh_close_to_exact_gelu(oracle):
    # The tanh form approximates x * Phi(x) within 4.8e-4 everywhere; a dropped
    # cubic term (3.4e-2) or a wrong constant breaks this.
    for x in np.linspace(-8, 8, 1601):
        exact = x * 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))
        assert abs(oracle.gelu_tanh(x) - exact) < 5e-4


def test_gelu_tanh_odd_part_and_special_values(oracle):
    # tanh is odd, so gelu(x) - gelu(-x) = x exactly in real arithmetic
    for x in (0.25, 0.5, 1.0, 2.5, 7.0):
        assert abs(oracle.gelu_tanh(x) - oracle.gelu_tanh(-x) - x) < 1e-15 * max(1.0, x)
    assert oracle.gelu_tanh(0.0) == 0.0
    assert oracle.gelu_tanh(50.0) == 50.0   # 1 + tanh(large) == 2


# ---------------------------------------------------------------- SiLU
def test_silu_matches_torch_and_identities(oracle):
    xs = np.linspace(-30, 30, 3001)
    ref = F.silu(torch.tensor(xs, dtype=torch.float64)).numpy()
    got = np.array([oracle.silu(x) for x in xs])
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0
    for x in (0.5, 1.0, 3.0, 10.0):
        assert abs(oracle.silu(x) - oracle.silu(-x) - x) < 1e-14 * max(1.0, x)


def test_silu_and_mul_against_library_and_rounding(oracle):
    x = W.silu(64, d=96)
    bits = W.to_bits(x)
    ref, ref16 = oracle.silu_and_mul(bits, d=96)
    xf = x.to(torch.float64)
    lib = (F.silu(xf[:, :96]) * xf[:, 96:]).numpy()
    assert np.allclose(ref, lib, rtol=1e-14, atol=1e-300)
    # ref16 is the nearest bf16 to ref: no other bf16 is strictly closer
    val = W.from_bits(ref16).to(torch.float64).numpy()
    up = W.from_bits((ref16.astype(np.int32) + np.where(ref16 & 0x8000, -1, 1)).astype(np.uint16))
    dn = W.from_bits((ref16.astype(np.int32) - np.where(ref16 & 0x8000, -1, 1)).astype(np.uint16))
    err = np.abs(val - ref)
    nz = ref16 & 0x7FFF != 0
    assert np.all(err[nz] <= np.abs(up.to(torch.float64).numpy() - ref)[nz])
    assert np.all(err[nz] <= np.abs(dn.to(torch.float64).numpy() - ref)[nz])


def test_silu_gate_is_first_half(oracle):
    # gate = [1, 0], up = [2, 5]: out = [silu(1) * 2, silu(0) * 5] = [2 silu(1), 0]
    x = torch.tensor([[1.0, 0.0, 2.0, 5.0]], dtype=torch.bfloat16)
    ref, _ = oracle.silu_and_mul(W.to_bits(x), d=2)
    s1 = F.silu(torch.tensor(1.0, dtype=torch.float64)).item()
    assert ref[0, 0] == pytest.approx(2 * s1, rel=1e-15)
    assert ref[0, 1] == 0.0


# ---------------------------------------------------------------- gelu_and_mul_sparse
def _run(oracle, rows, d, z, row_stride=None):
    x = torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)
    return oracle.gelu_and_mul_sparse(W.to_bits(x), d=d, z=z, row_stride=row_stride)


def test_worked_example_d2(oracle):
    # gate [1, 3], up [7, -2], z = 0.5: mean 2, population std 1, cutoff 2.5,
    # s = [0, 0.5]  ->  out = [0, gelu_tanh(0.5) * (-2)].
    res = _run(oracle, [[1.0, 3.0, 7.0, -2.0]], d=2, z=0.5)
    g05 = F.gelu(torch.tensor(0.5, dtype=torch.float64), approximate="tanh").item()
    assert res.mean[0] == 2.0 and res.std[0] == 1.0 and res.cutoff[0] == 2.5
    assert res.ref[0, 0] == 0.0
    assert res.ref[0, 1] == pytest.approx(-2.0 * g05, rel=1e-15)
    assert list(res.mask[0]) == [False, True]
    # with z = 1.645 > 1 the cutoff 3.645 is above both gates: all zero
    res = _run(oracle, [[1.0, 3.0, 7.0, -2.0]], d=2, z=Z95)
    assert np.all(res.ref == 0.0) and not res.mask.any()


def test_worked_example_d4(oracle):
    # gate [0, 0, 0, 4], up [1, 1, 1, 3], z = 1: mean 1, var (1+1+1+9)/4 = 3,
    # cutoff 1 + sqrt 3, s = [0, 0, 0, 3 - sqrt 3].
    res = _run(oracle, [[0, 0, 0, 4, 1, 1, 1, 3]], d=4, z=1.0)
    s = 3.0 - math.sqrt(3.0)
    want = 3.0 * F.gelu(torch.tensor(s, dtype=torch.float64), approximate="tanh").item()
    assert res.std[0] == pytest.approx(math.sqrt(3.0), rel=1e-15)
    assert np.all(res.ref[0, :3] == 0.0)
    assert res.ref[0, 3] == pytest.approx(want, rel=1e-14)


def test_d1_is_always_zero(oracle):
    # one gate value: std = 0, cutoff = the value itself, s = 0
    for g, u in ((3.0, 2.0), (-1.5, 4.0), (0.0, -1.0)):
        res = _run(oracle, [[g, u]], d=1, z=Z95)
        assert res.std[0] == 0.0 and res.ref[0, 0] == 0.0 and not res.mask.any()


def test_row_stats_are_mean_and_population_std(oracle):
    rng = np.random.default_rng(11)
    for T, d in ((7, 33), (3, 1000), (2, 4096)):
        x = torch.from_numpy(rng.standard_normal((T, 2 * d)).astype(np.float32) * 3 + 1).to(torch.bfloat16)
        res = oracle.gelu_and_mul_sparse(W.to_bits(x), d=d, z=0.3)
        g = x[:, :d].to(torch.float64).numpy()
        assert np.allclose(res.mean, g.mean(axis=1), rtol=1e-13, atol=1e-13)
        assert np.allclose(res.std, g.std(axis=1, ddof=0), rtol=1e-13)
        assert np.allclose(res.cutoff, res.mean + 0.3 * res.std, rtol=1e-15, atol=1e-15)


def test_constant_rows_give_exact_zero(oracle):
    inp = W.sweep(8, 2048, z=Z95, const_rows=True)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=inp.d, z=inp.z)
    for k, c in enumerate(W.CONST_GATES):
        r = inp.T - len(W.CONST_GATES) + k
        assert res.mean[r] == c and res.std[r] == 0.0 and res.cutoff[r] == c
        assert np.all(res.ref[r] == 0.0) and not res.mask[r].any()


def test_z0_cuts_at_the_mean(oracle):
    inp = W.iid(16, 1024, seed=9, z=0.0)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=inp.d, z=0.0)
    g = inp.x[:, :inp.d].to(torch.float64).numpy()
    assert np.array_equal(res.mask, g > g.mean(axis=1, keepdims=True))
    assert np.array_equal(res.ref != 0.0, res.mask & (inp.x[:, inp.d:].to(torch.float64).numpy() != 0))


@pytest.mark.parametrize("z,target", [(Z95, 0.95), (0.0, 0.5)])
def test_gaussian_zero_fraction_matches_target_sparsity(oracle, z, target):
    # On i.i.d. Gaussian rows the share of gates at or below mean + z std is
    # Phi(z); estimation noise at d = 16384 over 64 rows is ~1e-3.
    inp = W.iid(64, 16384, seed=123, z=z)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=inp.d, z=z)
    frac = 1.0 - res.mask.mean()
    assert abs(frac - target) < 0.003
    assert abs((res.ref == 0.0).mean() - target) < 0.003


def test_prefill_rows_zero_fraction(oracle):
    # per-row affine Gaussians: the threshold adapts to each row's mean/std
    inp = W.prefill(T=64)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=inp.d, z=inp.z)
    assert abs((1.0 - res.mask.mean()) - 0.95) < 0.003


def test_affine_invariance_of_the_mask(oracle):
    # g -> 2 g + 0.5 (exact in bf16 on small integers): mean -> 2 mean + 0.5,
    # std -> 2 std, so the mask is unchanged and s doubles.
    rng = np.random.default_rng(3)
    g = rng.integers(-8, 9, size=(32, 64)).astype(np.float32)
    u = rng.integers(-4, 5, size=(32, 64)).astype(np.float32)
    a = _run(oracle, np.concatenate([g, u], 1), d=64, z=0.7)
    b = _run(oracle, np.concatenate([2 * g + 0.5, u], 1), d=64, z=0.7)
    assert np.array_equal(a.mask, b.mask)
    s_a = np.maximum(g - a.cutoff[:, None], 0)
    s_b = np.maximum((2 * g + 0.5) - b.cutoff[:, None], 0)
    assert np.allclose(s_b, 2 * s_a, rtol=1e-12, atol=1e-12)


def _torch_composition(x: torch.Tensor, d: int, z: float) -> torch.Tensor:
    """Unfused fp64 composition of library ops (mean, population std, relu, tanh-GELU, mul)."""
    xf = x.to(torch.float64)
    g, u = xf[:, :d], xf[:, d:2 * d]
    mean = g.mean(dim=1, keepdim=True)
    std = g.std(dim=1, keepdim=True, unbiased=False)
    return F.gelu(torch.relu(g - (mean + std * z)), approximate="tanh") * u


def test_brute_force_small_integer_rows(oracle):
    # every gate row in {-2..2}^d for d = 1..4, against the library composition
    vals = np.array([-2.0, -1.0, 0.0, 1.0, 2.0])
    for d in range(1, 5):
        grid = np.stack(np.meshgrid(*([vals] * d), indexing="ij"), -1).reshape(-1, d)
        up = np.tile(np.arange(1, d + 1, dtype=np.float64) * 0.75 - 1.0, (len(grid), 1))
        x = torch.tensor(np.concatenate([grid, up], 1), dtype=torch.float32).to(torch.bfloat16)
        for z in (0.0, 0.5, Z95):
            res = oracle.gelu_and_mul_sparse(W.to_bits(x), d=d, z=z)
            want = _torch_composition(x, d, z).numpy()
            assert np.allclose(res.ref, want, rtol=1e-12, atol=1e-14), (d, z)


@pytest.mark.parametrize("T,d,rs,z", [(5, 31, 62, Z95), (3, 128, 300, 0.0), (9, 2048, 4096, Z95),
                                      (2, 33, 80, 1.0)])
def test_composition_on_random_rows(oracle, T, d, rs, z):
    inp = W.iid(T, d, seed=T * 31 + d, row_stride=rs)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=z, row_stride=rs)
    assert not np.isnan(res.ref).any()          # padding (NaN) is never read
    want = _torch_composition(inp.x, d, z).numpy()
    assert np.allclose(res.ref, want, rtol=1e-12, atol=1e-13)


def test_gate_is_first_half_and_up_second(oracle):
    # gate [0, 4] up [1, 9] vs the swapped layout: only the gate half sets the mask
    a = _run(oracle, [[0.0, 4.0, 1.0, 9.0]], d=2, z=0.0)
    assert list(a.mask[0]) == [False, True]
    assert a.ref[0, 1] == pytest.approx(
        9.0 * F.gelu(torch.tensor(2.0, dtype=torch.float64), approximate="tanh").item(), rel=1e-15)


def test_nan_gate_poisons_only_its_row(oracle):
    x = W.iid(3, 64, seed=1).x.clone()
    x[1, 5] = float("nan")
    res = oracle.gelu_and_mul_sparse(W.to_bits(x), d=64, z=Z95)
    assert np.isnan(res.ref[1]).all()
    assert not np.isnan(res.ref[[0, 2]]).any()


# ---------------------------------------------------------------- dense gelu_and_mul, squared_relu
def test_gelu_tanh_negative_tail_against_high_precision(oracle):
    # far-negative inputs, where 1 + tanh(y) cancels in double: compare with a
    # 50-digit evaluation of the defining expression
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 400
    k = mpmath.sqrt(2 / mpmath.pi)
    for x in (-3.0, -5.5, -8.0, -10.0, -12.5, -20.0):
        xm = mpmath.mpf(x)
        exact = 0.5 * xm * (1 + mpmath.tanh(k * (xm + mpmath.mpf("0.044715") * xm ** 3)))
        got = oracle.gelu_tanh(x)
        assert got == pytest.approx(float(exact), rel=1e-12, abs=0.0), x


def test_gelu_and_mul_dense_against_library(oracle):
    x = W.iid(33, 100, seed=8, row_stride=232).x
    ref, ref16 = oracle.gelu_and_mul(W.to_bits(x), d=100)
    xf = x[:, :200].to(torch.float64)
    lib = (F.gelu(xf[:, :100], approximate="tanh") * xf[:, 100:]).numpy()
    assert np.allclose(ref, lib, rtol=1e-12, atol=1e-15)
    # the bf16 copy is the nearest bf16 to ref (checked through torch on the
    # binary32 value, which is exact here only when ref is binary32-exact: use
    # the rounding property instead)
    val = W.from_bits(ref16).to(torch.float64).numpy()
    assert np.all(np.abs(val - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-38)


def test_gelu_and_mul_dense_gate_is_first_half(oracle):
    x = torch.tensor([[1.0, -1.0, 2.0, 3.0]], dtype=torch.bfloat16)
    ref, _ = oracle.gelu_and_mul(W.to_bits(x), d=2)
    g = F.gelu(torch.tensor([1.0, -1.0], dtype=torch.float64), approximate="tanh").numpy()
    assert np.allclose(ref[0], g * np.array([2.0, 3.0]), rtol=1e-15)


def test_squared_relu_against_library_exactly(oracle):
    rng = np.random.default_rng(12)
    x = torch.from_numpy(rng.standard_normal((17, 300)).astype(np.float32) * 4).to(torch.bfloat16)
    ref, ref16 = oracle.squared_relu_rows(W.to_bits(x))
    xf = x.to(torch.float64)
    assert np.array_equal(ref, (torch.relu(xf) ** 2).numpy())
    # x is bf16, so x^2 is exact in binary32 and torch's float -> bf16 cast is
    # the single correct rounding: the oracle's bits must match it
    t16 = (torch.relu(x.float()) ** 2).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ref16, t16)
    assert oracle.squared_relu(-0.5) == 0.0 and oracle.squared_relu(3.0) == 9.0
    assert np.isnan(oracle.squared_relu(float("nan")))


# ---------------------------------------------------------------- fp16 / fp32 elements
def test_f16_decode_matches_numpy_for_all_patterns(oracle):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.f16_to_double(0x0001) == 2.0 ** -24 and oracle.f16_to_double(0x7BFF) == 65504.0


@pytest.mark.parametrize("dt", [np.float16, np.float32])
def test_typed_sparse_gelu_matches_composition(oracle, dt):
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((9, 2 * 300 + 12)) * 1.5 + 0.3).astype(dt)
    res = oracle.gelu_and_mul_sparse_typed(x, d=300, z=1.2)
    want = _torch_composition(torch.from_numpy(x.astype(np.float64)), 300, 1.2).numpy()
    assert np.allclose(res.ref, want, rtol=1e-12, atol=1e-13)
    g = x[:, :300].astype(np.float64)
    assert np.allclose(res.std, g.std(axis=1), rtol=1e-13)


def test_typed_sparse_gelu_agrees_with_bf16_path_on_bf16_values(oracle):
    # bf16 values are exactly representable in fp32: the fp32 path must give
    # the same result as the bf16 path on the same values
    inp = W.iid(7, 512, seed=3)
    a = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=512, z=inp.z)
    b = oracle.gelu_and_mul_sparse_typed(inp.x.float().numpy(), d=512, z=inp.z)
    assert np.array_equal(a.ref, b.ref) and np.array_equal(a.mask, b.mask)


def test_typed_worked_example_fp32(oracle):
    x = np.array([[1.0, 3.0, 7.0, -2.0]], dtype=np.float32)
    res = oracle.gelu_and_mul_sparse_typed(x, d=2, z=0.5)
    g05 = F.gelu(torch.tensor(0.5, dtype=torch.float64), approximate="tanh").item()
    assert res.ref[0, 0] == 0.0 and res.ref[0, 1] == pytest.approx(-2.0 * g05, rel=1e-15)


# ---------------------------------------------------------------- native-rounding mode
def test_round_f16_matches_numpy(oracle):
    rng = np.random.default_rng(8)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
                        [65504.0, 65519.9, 65520.0, 6e-8, 3e-8, 2.98e-8, -1e-9, 0.0]])
    # numpy rounds float64 -> float16 directly (one rounding); the values past
    # 65520 overflow to infinity on purpose
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).astype(np.float64)
    got = np.array([oracle.round_f16(x) for x in v])
    assert np.array_equal(got, want)


def test_native_mode_against_torch_cpu_composition(oracle):
    # The native-rounding oracle (each op exact, rounded to the element type)
    # against torch's own CPU composition of the separate ops in that type.
    # fp32 accumulation order in torch's mean/std can move a rounded statistic
    # by one step on rare rows; everywhere else the two agree exactly.
    for dt in (torch.bfloat16, torch.float16):
        x = W.prefill(T=48, d=4096, dtype=dt).x
        g, u = x[:, :4096], x[:, 4096:]
        m = g.mean(dim=1, keepdim=True)
        sd = g.std(dim=1, keepdim=True, unbiased=False)
        c = m + sd * Z95
        want = (F.gelu(torch.relu(g - c), approximate="tanh") * u).to(torch.float64).numpy()
        arr = W.to_bits(x) if dt == torch.bfloat16 else x.numpy()
        ref, mask, cut = oracle.gelu_and_mul_sparse_native(arr, d=4096, z=Z95,
                                                           bf16_bits=dt == torch.bfloat16)
        same_rows = cut == c.to(torch.float64).numpy()[:, 0]
        assert same_rows.mean() >= 0.95
        # where the rounded cutoff agrees, every element agrees bit for bit
        assert np.array_equal(ref[same_rows], want[same_rows])


def test_native_mode_worked_example(oracle):
    # gate [1, 3], up [7, -2], z = 0.5 in bf16: m = 2, sd = 1, t = R(0.5) = 0.5,
    # c = 2.5; s = R(3 - 2.5) = 0.5; a = R(gelu(0.5)) ; out = R(a * -2)
    x = torch.tensor([[1.0, 3.0, 7.0, -2.0]], dtype=torch.bfloat16)
    ref, mask, cut = oracle.gelu_and_mul_sparse_native(W.to_bits(x), d=2, z=0.5, bf16_bits=True)
    a = torch.tensor(F.gelu(torch.tensor(0.5, dtype=torch.float64), approximate="tanh").item(),
                     dtype=torch.float64).to(torch.bfloat16).to(torch.float64).item()
    want = torch.tensor(a * -2.0, dtype=torch.float64).item()
    assert cut[0] == 2.5 and ref[0, 0] == 0.0 and list(mask[0]) == [False, True]
    assert ref[0, 1] == oracle.round_bf16(want)


def test_native_mode_rounds_the_statistics(oracle):
    # a row whose exact mean is not a bf16 number: the cutoff must be built
    # from the rounded mean (0.333... -> 0.333984375), not the exact one
    x = torch.tensor([[0.0, 0.0, 1.0, 1.0, 1.0, 1.0]], dtype=torch.bfloat16)
    ref, mask, cut = oracle.gelu_and_mul_sparse_native(W.to_bits(x), d=3, z=0.0, bf16_bits=True)
    assert cut[0] == oracle.round_bf16(1.0 / 3.0) == 0.333984375
