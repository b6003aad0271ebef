"""Build the CUDA library ``gated_activation_gb300/_lib/libgated_act.so`` in-tree.

One nvcc per translation unit, run in parallel, then one shared-library link.
Target: sm_103a only (``-gencode arch=compute_103a,code=sm_103a``), with
``-lineinfo`` for the profiler and the CUDA runtime linked statically so the
library loads wherever the driver does.  No fast-math: the statistics use
IEEE division and square root.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libgated_act.so")
SOURCES = ("api.cu", "gelu_and_mul_sparse.cu", "elementwise.cu")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def cflags(extra: list[str] | None = None) -> list[str]:
    return [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC] + (extra or [])


def _compile(src: str, obj: str, extra: list[str]) -> tuple[str, str]:
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + cflags(extra)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{r.stderr}")
    return src, r.stderr


def build(verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile all sources and link the shared library; returns its path."""
    extra = list(extra or [])
    os.makedirs(LIB_DIR, exist_ok=True)
    with tempfile.TemporaryDirectory(dir=LIB_DIR) as tmp:
        objs = [os.path.join(tmp, s.replace(".cu", ".o")) for s in SOURCES]
        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            for src, err in ex.map(lambda a: _compile(*a, extra), zip(SOURCES, objs)):
                if verbose and err:
                    print(f"[{src}]\n{err}", file=sys.stderr)
        out_tmp = os.path.join(tmp, "libgated_act.so")
        cmd = [nvcc(), "-shared", ARCH, "-cudart", "static", "-o", out_tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stderr}")
        os.replace(out_tmp, LIB)
    return LIB


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return all(os.path.getmtime(p) <= t for p in deps)


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(verbose=v, extra=["-Xptxas", "-v"] if v else None))
