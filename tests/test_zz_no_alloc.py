"""The no-allocation entry point, gelu_and_mul_sparse_ws_static.

Callers that cannot allocate device memory (an engine that reserved all free
memory for its own pool, a plugin host that passes only inputs and outputs)
use this variant: its row counters live in a small scratch array inside the
library instead of a caller workspace.  This file is collected last.  The test
calls the entry point through the C ABI twice in a row and checks each output
against the plain entry point within the bf16 tolerance of the other tests.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import ATOL, RTOL

pytestmark = pytest.mark.gpu


def _close(a: torch.Tensor, b: torch.Tensor) -> bool:
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    if not np.array_equal(np.isnan(x), np.isnan(y)):
        return False
    ok = np.isnan(y) | (np.abs(x - y) <= RTOL * np.abs(y) + ATOL)
    return bool(ok.all())


# (T, d, variant): rows taken dynamically through the static scratch (the
# first two), and a geometry that needs no scratch
CASES = [(2048, 16384, 0), (700, 8192, 4), (64, 4096, 0)]


def test_static_scratch_entry_matches_plain_entry_twice():
    ga = require_gpu()
    lib = ga.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for T, d, variant in CASES:
        x = W.iid(T, d, seed=T + d).x.cuda()
        ref = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        rc = lib.gelu_and_mul_sparse(ref.data_ptr(), x.data_ptr(), T, d, 2 * d, W.Z95, stream)
        assert rc == ga.OK
        for call in range(2):          # two calls in a row share the scratch array
            out = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
            rc = lib.gelu_and_mul_sparse_ws_static(out.data_ptr(), x.data_ptr(), T, d, 2 * d,
                                                   W.Z95, ga.BF16, variant, 0, stream)
            assert rc == ga.OK, ga.status_string(rc)
            torch.cuda.synchronize()
            assert _close(out, ref), f"T={T} d={d} call {call}"
