"""The oracle's pins have teeth: planted mistakes must fail at least one pin.

Each case copies the oracle's C source to a temporary directory, plants one
plausible slip by a textual substitution (a sign, a dropped term, sample
instead of population variance, the wrong half, no relu, a non-strict mask,
truncation instead of round-to-nearest-even ...), compiles that copy and runs
a battery of the independent checks.  The committed oracle is never touched.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import workloads as W

SRC = os.path.join(os.path.dirname(O.__file__), "gated_act_oracle.c")

MUTANTS = {
    "cutoff_sign": ("double cutoff = mean + std * z;", "double cutoff = mean - std * z;"),
    "sample_variance": ("double var = ss / (double)d;", "double var = ss / (double)(d - 1);"),
    "std_is_variance": ("double std = sqrt(var);", "double std = var;"),
    "mean_divisor": ("\n        double mean = sum / (double)d;",
                     "\n        double mean = sum / (double)(d + 1);"),
    "dropped_cubic": ("(x + 0.044715 * x * x * x)", "(x)"),
    "cubic_is_square": ("0.044715 * x * x * x", "0.044715 * x * x"),
    "gelu_scale": ("sqrt(2.0 / ORACLE_PI)", "sqrt(1.0 / ORACLE_PI)"),
    "multiplies_gate": ("ref[r * d + j] = oracle_gelu_tanh(s) * u;",
                        "ref[r * d + j] = oracle_gelu_tanh(s) * g;"),
    "no_relu": ("if (s < 0.0)\n                s = 0.0;", ""),
    "gelu_unshifted": ("ref[r * d + j] = oracle_gelu_tanh(s) * u;",
                       "ref[r * d + j] = (s > 0.0 ? oracle_gelu_tanh(g) : 0.0) * u;"),
    "mask_not_strict": ("(uint8_t)(g > cutoff)", "(uint8_t)(g >= cutoff)"),
    "up_offset": ("const int64_t g0 = r * row_stride, u0 = g0 + d;",
                  "const int64_t g0 = r * row_stride, u0 = g0 + d - 1;"),
    "f16_exponent_bias": ("v = ldexp((double)(f + 1024), e - 25);",
                          "v = ldexp((double)(f + 1024), e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "f32_read_as_f16": ("    if (dtype == ORACLE_F32) {", "    if (dtype == -1) {"),
    "encode_truncates": ("double r = rint(a / q) * q;", "double r = floor(a / q) * q;"),
    "encode_via_float": ("double r = rint(a / q) * q;",
                         "double r = rint((double)(float)a / q) * q;"),
    "silu_sign": ("return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    "gelu_negative_branch": ("return x * t / (1.0 + t);", "return x * t / (1.0 - t);"),
    "gelu_negative_exponent": ("const double t = exp(2.0 * y);", "const double t = exp(y);"),
    "squared_relu_not_squared": ("    return r * r;", "    return r;"),
    "squared_relu_keeps_negative": ("double r = x > 0.0 ? x : 0.0;", "double r = x;"),
    "dense_gelu_uses_up_twice": ("double y = oracle_gelu_tanh(oracle_bf16_to_double(gate[j])) *\n"
                                 "                       oracle_bf16_to_double(up[j]);\n"
                                 "            if (ref)\n                ref[r * d + j] = y;\n"
                                 "            if (ref_bf16)\n                ref_bf16[r * d + j] = oracle_double_to_bf16(y);\n"
                                 "        }\n    }\n    return 0;\n}\n\n/*\n * squared_relu",
                                 "double y = oracle_gelu_tanh(oracle_bf16_to_double(up[j])) *\n"
                                 "                       oracle_bf16_to_double(up[j]);\n"
                                 "            if (ref)\n                ref[r * d + j] = y;\n"
                                 "            if (ref_bf16)\n                ref_bf16[r * d + j] = oracle_double_to_bf16(y);\n"
                                 "        }\n    }\n    return 0;\n}\n\n/*\n * squared_relu"),
    "native_no_stat_rounding": ("const double m = R(mean);", "const double m = mean;"),
    "native_unrounded_shift": ("double s = R(g - c);", "double s = g - c;"),
    "native_no_product_rounding": ("ref[r * d + j] = R(a * u);", "ref[r * d + j] = a * u;"),
    "f16_round_subnormal_scale": ("    if (e < -14)\n        e = -14;", "    if (e < -15)\n        e = -15;"),
    "silu_up_is_gate": ("double y = oracle_silu(oracle_bf16_to_double(gate[j])) *\n"
                        "                       oracle_bf16_to_double(up[j]);",
                        "double y = oracle_silu(oracle_bf16_to_double(gate[j])) *\n"
                        "                       oracle_bf16_to_double(gate[j]);"),
}


def _composition(x, d, z):
    xf = x.to(torch.float64)
    g, u = xf[:, :d], xf[:, d:2 * d]
    mean = g.mean(dim=1, keepdim=True)
    std = g.std(dim=1, keepdim=True, unbiased=False)
    return F.gelu(torch.relu(g - (mean + std * z)), approximate="tanh") * u


def _battery(o: O.Oracle) -> dict:
    """Independent checks; True = passes."""
    out = {}
    xs = np.linspace(-3, 10, 261)
    ref = F.gelu(torch.tensor(xs, dtype=torch.float64), approximate="tanh").numpy()
    out["gelu_vs_torch"] = bool(np.allclose([o.gelu_tanh(x) for x in xs], ref, rtol=1e-13))
    sx = np.linspace(-20, 20, 81)
    out["silu_vs_torch"] = bool(np.allclose([o.silu(x) for x in sx],
                                            F.silu(torch.tensor(sx)).numpy(), rtol=1e-13))
    inp = W.iid(6, 40, seed=4)
    res = o.gelu_and_mul_sparse(W.to_bits(inp.x), d=40, z=0.4)
    out["composition"] = bool(np.allclose(res.ref, _composition(inp.x, 40, 0.4).numpy(),
                                          rtol=1e-12, atol=1e-13))
    g = inp.x[:, :40].to(torch.float64).numpy()
    out["mask_vs_numpy"] = bool(np.array_equal(
        res.mask, g > (g.mean(1) + 0.4 * g.std(1))[:, None]))
    c = W.sweep(1, 64, const_rows=True)
    rc = o.gelu_and_mul_sparse(W.to_bits(c.x), d=64, z=W.Z95)
    out["constant_rows"] = bool(np.all(rc.ref[1:] == 0.0) and not rc.mask[1:].any())
    big = W.iid(16, 8192, seed=77)
    rb = o.gelu_and_mul_sparse(W.to_bits(big.x), d=8192, z=W.Z95)
    out["zero_fraction"] = abs((1 - rb.mask.mean()) - 0.95) < 0.003
    f = np.random.default_rng(1).standard_normal(4000).astype(np.float32)
    tb = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out["encode_vs_torch"] = bool(np.array_equal([o.double_to_bf16(float(v)) for v in f], tb))
    out["encode_once"] = o.double_to_bf16(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    s = W.silu(8, d=32)
    r64, r16 = o.silu_and_mul(W.to_bits(s), d=32)
    sf = s.to(torch.float64)
    out["silu_and_mul_vs_torch"] = bool(np.allclose(r64, (F.silu(sf[:, :32]) * sf[:, 32:]).numpy(),
                                                    rtol=1e-13, atol=1e-300))
    xs = np.linspace(-9, 3, 97)
    out["gelu_negative_tail"] = bool(np.allclose(
        [o.gelu_tanh(x) for x in xs],
        F.gelu(torch.tensor(xs), approximate="tanh").numpy(), rtol=1e-10, atol=1e-13))
    dx = W.iid(5, 24, seed=6).x
    g64, _ = o.gelu_and_mul(W.to_bits(dx), d=24)
    dxf = dx.to(torch.float64)
    out["dense_gelu_vs_torch"] = bool(np.allclose(
        g64, (F.gelu(dxf[:, :24], approximate="tanh") * dxf[:, 24:]).numpy(), rtol=1e-12,
        atol=1e-15))
    q64, _ = o.squared_relu_rows(W.to_bits(dx))
    out["squared_relu_vs_torch"] = bool(np.array_equal(q64, (torch.relu(dxf) ** 2).numpy()))
    hb = np.arange(0, 1 << 16, 64, dtype=np.uint32).astype(np.uint16)
    hv = hb.view(np.float16).astype(np.float64)
    hg = np.array([o.f16_to_double(int(b)) for b in hb])
    fin = np.isfinite(hv)
    out["f16_decode_vs_numpy"] = bool(np.array_equal(hg[fin], hv[fin]))
    x32 = (np.random.default_rng(2).standard_normal((3, 80)) * 2).astype(np.float32)
    t32 = o.gelu_and_mul_sparse_typed(x32, d=40, z=0.4)
    out["typed_f32_vs_torch"] = bool(np.allclose(
        t32.ref, _composition(torch.from_numpy(x32.astype(np.float64)), 40, 0.4).numpy(),
        rtol=1e-12, atol=1e-13))
    v = np.random.default_rng(4).standard_normal(3000) * 1e-5
    out["round_f16_vs_numpy"] = bool(np.array_equal(
        [o.round_f16(t) for t in v], v.astype(np.float16).astype(np.float64)))
    nx = W.prefill(T=128, d=512, dtype=torch.bfloat16).x
    ng, nu = nx[:, :512], nx[:, 512:]
    nc = ng.mean(1, keepdim=True) + ng.std(1, keepdim=True, unbiased=False) * 1.3
    nwant = (F.gelu(torch.relu(ng - nc), approximate="tanh") * nu).to(torch.float64).numpy()
    nref, _, ncut = o.gelu_and_mul_sparse_native(W.to_bits(nx), d=512, z=1.3, bf16_bits=True)
    same = ncut == nc.to(torch.float64).numpy()[:, 0]
    out["native_vs_torch"] = bool(same.mean() >= 0.95 and np.array_equal(nref[same], nwant[same]))
    out["silu_rounded"] = bool(np.all(
        np.abs(W.from_bits(r16).to(torch.float64).numpy() - r64) <= np.abs(r64) * 2.0 ** -8 + 1e-38))
    return out


def test_battery_passes_on_the_committed_oracle():
    res = _battery(O.default())
    assert all(res.values()), res


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    # the first occurrence is the one planted (the fp64 definition comes
    # before the native-rounding composition in the source)
    assert src.count(old) >= 1, f"mutation anchor for {name} not present"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = O.build.compile_oracle(str(mutated), str(tmp_path / "libmutant.so"), openmp=False)
    res = _battery(O.Oracle(lib))
    failed = [k for k, ok in res.items() if not ok]
    assert failed, f"mutant {name} passed every pin"
