"""The no-allocation entry point, gelu_and_mul_sparse_ws_static.

Some callers cannot allocate device memory: an inference engine that reserved
all free memory for its own pool at start-up, or a plugin host that passes a
kernel only its inputs and outputs.  They call this variant, whose row
counters live in a small scratch array inside the library instead of a
workspace the caller allocates.

The test calls the entry point through the C ABI twice in a row on each case
(both calls share the array).  Every output is checked against the fp64
oracle with the acceptance criteria of the other GPU tests, and bitwise
against gelu_and_mul_sparse_ws given a fresh zeroed workspace, which plans
the same geometry.  The plan query asserts which cases take rows from the
counters (and so use the array) and which need no scratch.  This file is
collected last, so a run that stops at the first failure has run every other
test before it.
"""
import ctypes

import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu

# (T, d, variant, rows taken from the counters): the first two use the array
# (pipe rows at the prefill shape; forced tma rows, ragged against the grid),
# the third plans one CTA per row and needs no scratch
CASES = [(2048, 16384, 0, 1), (700, 8192, 4, 1), (64, 4096, 0, 0)]


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().view(torch.int16)


def test_static_scratch_entry_matches_oracle_and_workspace_entry_twice(oracle):
    ga = require_gpu()
    lib = ga.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for T, d, variant, dynamic in CASES:
        inp = W.iid(T, d, seed=T + d)
        x = inp.x.cuda()
        plan = ga.Plan()
        rc = lib.gelu_and_mul_sparse_plan_ex(0, x.data_ptr(), T, d, 2 * d, ga.BF16, variant, 0,
                                             0, 1, ctypes.byref(plan))
        assert rc == ga.OK
        assert plan.dynamic_rows == dynamic, (T, d, plan.as_dict())

        ws = ga.new_workspace()
        ref = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        rc = lib.gelu_and_mul_sparse_ws(ref.data_ptr(), x.data_ptr(), T, d, 2 * d, inp.z,
                                        ga.BF16, variant, 0, ws.data_ptr(), stream)
        assert rc == ga.OK, ga.status_string(rc)
        res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
        for call in range(2):          # two calls in a row share the scratch array
            out = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
            rc = lib.gelu_and_mul_sparse_ws_static(out.data_ptr(), x.data_ptr(), T, d, 2 * d,
                                                   inp.z, ga.BF16, variant, 0, stream)
            assert rc == ga.OK, ga.status_string(rc)
            torch.cuda.synchronize()
            check_gelu(out.cpu(), inp.x, d, res, f"static scratch T{T} d{d} call {call}")
            assert torch.equal(_bits(out), _bits(ref)), f"T={T} d={d} call {call}"
        assert int(ws.count_nonzero().item()) == 0
