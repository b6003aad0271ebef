"""Golden fixtures: oracle regression values and numbers printed on the pages."""
import json
import os

import numpy as np
import pytest

import workloads as W

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def test_oracle_matches_its_regression_fixture(oracle):
    import hashlib
    gold = _load("oracle_regression.json")["cases"]
    inputs = {"tiny": W.tiny(), "sweep_T8_d2048": W.sweep(8, 2048, z=0.0), "decode_T4": W.decode(4)}
    for name, inp in inputs.items():
        g = gold[name]
        bits = W.to_bits(inp.x)
        assert hashlib.sha256(bits.tobytes()).hexdigest() == g["input_sha256"], \
            f"{name}: the seeded generator no longer reproduces the fixture's input"
        res = oracle.gelu_and_mul_sparse(bits, d=inp.d, z=inp.z)
        assert np.allclose(res.mean, g["row_mean"], rtol=0, atol=1e-15)
        assert np.allclose(res.std, g["row_std"], rtol=1e-15)
        assert np.allclose(res.cutoff, g["row_cutoff"], rtol=1e-15)
        assert int((res.ref != 0).sum()) == g["nonzero_count"]
        assert res.ref.sum() == pytest.approx(g["ref_sum"], rel=1e-12)
    s = W.silu(1024)
    _, r16 = oracle.silu_and_mul(W.to_bits(s))
    assert hashlib.sha256(r16.tobytes()).hexdigest() == gold["silu_M1024"]["ref_bf16_sha256"]


def test_target_sparsity_constant_matches_page_reading():
    p = _load("page_numbers.json")["sparse_gelu_target_sparsity"]
    assert p["z"] == W.Z95
