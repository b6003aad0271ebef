"""Randomised GPU parity of gelu_and_mul_sparse (and of its native-rounding mode).

Seeded draws of everything the launch depends on are each checked against the
fp64 oracle with the per-type tolerance of tests/parity.py:
- the row count, the width and the padding of the rows (NaN-filled);
- the threshold z (including negative values);
- the element type;
- a forced geometry (warp, CTA or cluster rows, scalar, bulk-copy or
  producer/consumer rows with a forced number of CTAs per SM) or the
  library's own choice;
- a workspace (dynamic rows) or none;
- a constant-gate row, whose output must be exactly zero.

A forced geometry that does not fit the draw must be refused with
GATED_ACT_ERR_VARIANT; the library's own choice never is.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu

# GATED_ACT_FUZZ_SCALE=k runs k times as many draws (the first ones unchanged)
SCALE = max(1, int(os.environ.get("GATED_ACT_FUZZ_SCALE", "1")))
N_CASES = 200 * SCALE
MAX_ELEMS = 3_000_000          # T * d per case, so the oracle stays fast
DTYPES = (torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.float16, torch.float32)
ELEM = {torch.bfloat16: 2, torch.float16: 2, torch.float32: 4}


@pytest.fixture(scope="module")
def ga():
    return require_gpu()


def draw(i: int, variants=(0, 0, 0, 1, 2, 2, 3, 4, 4), seed0: int = 20_000) -> dict:
    r = np.random.default_rng(seed0 + i)
    dt = DTYPES[int(r.integers(len(DTYPES)))]
    epv = 16 // ELEM[dt]
    if r.random() < 0.75:                      # the 16-byte layout
        d = epv * int(np.exp(r.uniform(0.0, np.log(32768 // epv))))
        pad = epv * int(r.integers(0, 3))
    else:                                      # anything else: the scalar path
        d = int(np.exp(r.uniform(0.0, np.log(20000))))
        pad = int(r.integers(0, 9))
    d = max(d, 1)
    t_max = max(1, MAX_ELEMS // d)
    T = int(min(t_max, np.exp(r.uniform(0.0, np.log(4096)))))
    T = max(T, 1)
    z = float(r.choice([0.0, W.Z95, r.uniform(-1.0, 3.0)]))
    variant = int(r.choice(list(variants)))
    cluster = 0
    if variant == 2:
        cluster = int(r.choice([0, 1, 2, 4, 8]))
    elif variant == 4:
        cluster = int(r.choice([0, 1, 2, 4, 8, 16]))
    elif variant == 5:
        cluster = int(r.choice([0, 0, 1, 2, 4, 8]))
    elif variant == 6:
        cluster = int(r.choice([2, 4, 8]))
    return {"dtype": dt, "T": T, "d": d, "rs": 2 * d + pad, "z": z, "variant": variant,
            "cluster": cluster, "ws": bool(r.random() < 0.5), "const_row": bool(r.random() < 0.5),
            "seed": 30_000 + i}


def oracle_result(oracle, x: torch.Tensor, d: int, z: float):
    if x.dtype == torch.bfloat16:
        return oracle.gelu_and_mul_sparse(W.to_bits(x), d=d, z=z)
    return oracle.gelu_and_mul_sparse_typed(x.contiguous().numpy(), d=d, z=z)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_launch(ga, oracle, i):
    run_case(ga, oracle, draw(i), f"case {i}")


# the producer/consumer geometry, forced (or the library's choice)
N_PIPE = 80 * SCALE


@pytest.mark.parametrize("i", range(N_PIPE))
def test_random_pipe_launch(ga, oracle, i):
    run_case(ga, oracle, draw(i, variants=(5, 5, 5, 0), seed0=90_000), f"pipe case {i}")


# split rows forced (or the library's choice)
N_SPLIT = 60 * SCALE


@pytest.mark.parametrize("i", range(N_SPLIT))
def test_random_split_launch(ga, oracle, i):
    run_case(ga, oracle, draw(i, variants=(6, 6, 6, 0), seed0=120_000), f"split case {i}")


def run_case(ga, oracle, c: dict, name: str):
    T, d, z = c["T"], c["d"], c["z"]
    inp = W.iid(T, d, seed=c["seed"], row_stride=c["rs"], z=z, dtype=c["dtype"])
    x = inp.x.clone()
    if c["const_row"]:
        x[T // 2, :d] = 0.75                   # exact in every element type: std = 0
    label = f"{name}: {c}"
    ws = ga.new_workspace() if c["ws"] else None
    try:
        out = ga.gelu_and_mul_sparse(x.cuda(), z, d=d, variant=c["variant"],
                                     cluster=c["cluster"], workspace=ws)
    except ga.GatedActError as e:
        assert c["variant"] != 0 and e.status == ga.ERR_VARIANT, label
        return
    torch.cuda.synchronize()
    if ws is not None:
        assert int(ws.count_nonzero().item()) == 0, label
    out = out.cpu()
    check_gelu(out, x, d, oracle_result(oracle, x, d, z), label)
    if c["const_row"]:
        assert torch.count_nonzero(out[T // 2].float()).item() == 0, label


# ------------------------------------------------------------ native-rounding mode
N_NATIVE = 60 * SCALE


def draw_native(i: int) -> dict:
    r = np.random.default_rng(60_000 + i)
    dt = (torch.bfloat16, torch.float16)[int(r.integers(2))]
    if r.random() < 0.75:
        d = 8 * int(np.exp(r.uniform(0.0, np.log(4096))))
        pad = 8 * int(r.integers(0, 3))
    else:
        d = int(np.exp(r.uniform(0.0, np.log(20000))))
        pad = int(r.integers(0, 9))
    d = max(d, 1)
    T = max(1, int(min(MAX_ELEMS // d, np.exp(r.uniform(0.0, np.log(2048))))))
    z = float(r.choice([0.0, W.Z95, 1.3, r.uniform(-1.0, 3.0)]))
    return {"dtype": dt, "T": T, "d": d, "rs": 2 * d + pad, "z": z, "seed": 70_000 + i}


@pytest.mark.parametrize("i", range(N_NATIVE))
def test_random_native_launch(ga, oracle, i):
    from tests.parity import check_native
    c = draw_native(i)
    T, d, z = c["T"], c["d"], c["z"]
    x = W.iid(T, d, seed=c["seed"], row_stride=c["rs"], z=z, dtype=c["dtype"]).x
    arr = W.to_bits(x) if x.dtype == torch.bfloat16 else x.contiguous().numpy()
    ref, mask, cut = oracle.gelu_and_mul_sparse_native(arr, d=d, z=z,
                                                       bf16_bits=x.dtype == torch.bfloat16)
    out = ga.gelu_and_mul_sparse_native(x.cuda(), z, d=d)
    torch.cuda.synchronize()
    check_native(out.cpu(), x, d, ref, mask, cut, f"native case {i}: {c}", z=z)
