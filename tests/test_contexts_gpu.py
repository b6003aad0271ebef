"""The library in contexts other than the device's primary one.

Some per-device state of the library belongs to one CUDA context: the
opt-in to more than 48 KB of shared memory for the bulk-copy kernels, the
address of the no-allocation entry point's scratch array, and the native
table.  A process that makes its own driver contexts current must see each
of them set up again in each context.

A fresh process (the driver API through ctypes, no PyTorch on the GPU)
creates two contexts on device 0 and, in each and then in the primary
context, runs through the C ABI:
  * forced pipe rows (the shared-memory opt-in),
  * the no-allocation entry point on pipe rows (the scratch array),
  * native-rounding rows (the table).
Every context must return the same bits, and those bits must pass the
oracle (pipe rows) or equal this process's own native call.  All three
contexts stay alive until the end, so no context handle is reused.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import require_gpu
from tests.parity import check_gelu

pytestmark = pytest.mark.gpu

PIPE = (8, 32768)      # T, d for the forced pipe-rows calls
NATIVE = (4, 4096)

_CHILD = r"""
import ctypes, os, sys
import numpy as np
sys.path.insert(0, {root!r})
import workloads as W
from gated_activation_gb300 import LIB_PATH

out_dir = {out_dir!r}
cu = ctypes.CDLL("libcuda.so.1")
lib = ctypes.CDLL(LIB_PATH)
i64, vp, dbl, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
lib.gelu_and_mul_sparse_ex.argtypes = [vp, vp, i64, i64, i64, dbl, ci, ci, vp]
lib.gelu_and_mul_sparse_ws_static.argtypes = [vp, vp, i64, i64, i64, dbl, ci, ci, ci, vp]
lib.gelu_and_mul_sparse_native.argtypes = [vp, vp, i64, i64, i64, dbl, ci, vp]


def ok(rc, what):
    if rc != 0:
        raise SystemExit(f"{{what}}: {{rc}}")


ok(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ok(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")


def make_context():
    ctx = ctypes.c_void_p()
    if hasattr(cu, "cuCtxCreate_v2"):
        ok(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate")
    else:
        ok(cu.cuCtxCreate_v4(ctypes.byref(ctx), None, 0, dev), "cuCtxCreate")
    return ctx


def run_all(tag):
    results = {{}}
    for name, (T, d) in (("pipe", {pipe}), ("static", {pipe}), ("native", {native})):
        x = W.to_bits(W.iid(T, d, seed=T + d).x)
        nin, nout = x.nbytes, T * d * 2
        din, dout = ctypes.c_uint64(), ctypes.c_uint64()
        ok(cu.cuMemAlloc_v2(ctypes.byref(din), ctypes.c_size_t(nin)), "cuMemAlloc")
        ok(cu.cuMemAlloc_v2(ctypes.byref(dout), ctypes.c_size_t(nout)), "cuMemAlloc")
        ok(cu.cuMemcpyHtoD_v2(din, x.ctypes.data_as(vp), ctypes.c_size_t(nin)), "HtoD")
        ok(cu.cuMemsetD8_v2(dout, 0xFF, ctypes.c_size_t(nout)), "memset")
        i, o, z = vp(din.value), vp(dout.value), W.Z95
        if name == "pipe":
            rc = lib.gelu_and_mul_sparse_ex(o, i, T, d, 2 * d, z, 5, 0, None)
        elif name == "static":
            rc = lib.gelu_and_mul_sparse_ws_static(o, i, T, d, 2 * d, z, 0, 5, 0, None)
        else:
            rc = lib.gelu_and_mul_sparse_native(o, i, T, d, 2 * d, z, 0, None)
        ok(rc, f"{{tag}} {{name}}")
        ok(cu.cuCtxSynchronize(), "sync")
        y = np.empty((T, d), dtype=np.uint16)
        ok(cu.cuMemcpyDtoH_v2(y.ctypes.data_as(vp), dout, ctypes.c_size_t(nout)), "DtoH")
        ok(cu.cuMemFree_v2(din), "free")
        ok(cu.cuMemFree_v2(dout), "free")
        np.save(os.path.join(out_dir, f"{{tag}}_{{name}}.npy"), y)


a = make_context()          # created current
run_all("ctx_a")
b = make_context()          # a second live context on the same device
run_all("ctx_b")
prim = ctypes.c_void_p()
ok(cu.cuDevicePrimaryCtxRetain(ctypes.byref(prim), dev), "retain")
ok(cu.cuCtxSetCurrent(prim), "set primary")
run_all("primary")
ok(cu.cuCtxSetCurrent(None), "unset")
ok(cu.cuCtxDestroy_v2(b), "destroy b")
ok(cu.cuCtxDestroy_v2(a), "destroy a")
ok(cu.cuDevicePrimaryCtxRelease_v2(dev), "release")
print("DONE")
"""


def test_every_context_sets_up_its_own_state(oracle, tmp_path):
    ga = require_gpu()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = _CHILD.format(root=root, out_dir=str(tmp_path), pipe=PIPE, native=NATIVE)
    r = subprocess.run([sys.executable, "-c", src], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0, (r.stdout[-1000:], r.stderr[-2000:])
    assert r.stdout.strip().endswith("DONE"), r.stdout[-500:]

    def load(tag, name):
        return np.load(tmp_path / f"{tag}_{name}.npy")

    for name in ("pipe", "static", "native"):
        first = load("ctx_a", name)
        for tag in ("ctx_b", "primary"):
            assert np.array_equal(first, load(tag, name)), (name, tag)

    T, d = PIPE
    inp = W.iid(T, d, seed=T + d)
    res = oracle.gelu_and_mul_sparse(W.to_bits(inp.x), d=d, z=W.Z95)
    for name in ("pipe", "static"):
        out = torch.from_numpy(load("ctx_a", name).view(np.int16)).view(torch.bfloat16)
        check_gelu(out, inp.x, d, res, f"{name} in a created context")

    T, d = NATIVE
    x = W.iid(T, d, seed=T + d).x.cuda()
    mine = ga.gelu_and_mul_sparse_native(x, W.Z95).cpu().view(torch.int16).numpy()
    assert np.array_equal(load("ctx_a", "native").view(np.int16), mine)
