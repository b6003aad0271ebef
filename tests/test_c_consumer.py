"""The C ABI from plain C: tests/c_consumer/consumer.c includes
include/gated_act.h, links the library and the CUDA runtime, and calls
gelu_and_mul_sparse, gelu_and_mul_sparse_ws and silu_and_mul on buffers it
allocates itself.  On the CPU it must compile as strict C99 with every
warning an error (the CUDA headers are included as system headers); on a GPU
its outputs must match the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import check_gelu, check_silu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_consumer", "consumer.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path) -> str:
    from gated_activation_gb300 import build as gbuild
    if not gbuild.up_to_date():
        gbuild.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(str(tmp_path), "consumer")
    lib_dir = os.path.dirname(gbuild.LIB)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-lgated_act", "-Wl,-rpath," + lib_dir,
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stderr}"
    return exe


def test_consumer_compiles_as_c99(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_consumer_matches_oracle(tmp_path, oracle):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(tmp_path)
    T, d, M = 300, 4096, 2048
    inp = W.iid(T, d, seed=77)
    xs = W.silu(M)
    p = lambda name: os.path.join(str(tmp_path), name)  # noqa: E731
    W.to_bits(inp.x).tofile(p("gelu_in"))
    W.to_bits(xs).tofile(p("silu_in"))
    r = subprocess.run([exe, str(T), str(d), repr(inp.z), p("gelu_in"), p("gelu_out"),
                        p("gelu_ws_out"), str(M), p("silu_in"), p("silu_out")],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=inp.z)
    for name in ("gelu_out", "gelu_ws_out"):
        y = W.from_bits(np.fromfile(p(name), dtype=np.uint16).reshape(T, d))
        check_gelu(y, inp.x, d, res, f"C consumer {name}")
    _, ref16 = oracle.silu_and_mul(W.to_bits(xs))
    check_silu(W.from_bits(np.fromfile(p("silu_out"), dtype=np.uint16).reshape(M, 768)), ref16,
               "C consumer silu")
