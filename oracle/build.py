"""Compile the C oracle into ``oracle/_build/liboracle.so`` (test infrastructure).

Plain gcc, fp64, OpenMP over rows when the compiler has it.  No CUDA and no
code shared with the CUDA library.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gated_act_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def _cc() -> str:
    return os.environ.get("CC", "gcc")


def compile_oracle(src: str = SRC, out: str = LIB, openmp: bool = True) -> str:
    """Compile ``src`` to the shared library ``out`` and return its path.

    Strict IEEE double arithmetic: -O2 without -ffast-math, and
    -ffp-contract=off so that no multiply-add is fused behind the source's back.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = [_cc(), "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-Wall", "-Wextra", src, "-o"]
    tmp = tempfile.NamedTemporaryFile(dir=os.path.dirname(out), suffix=".so",
                                      delete=False)
    tmp.close()
    try:
        if openmp:
            r = subprocess.run(base + [tmp.name, "-fopenmp", "-lm"],
                               capture_output=True, text=True)
            if r.returncode == 0:
                os.replace(tmp.name, out)
                return out
        r = subprocess.run(base + [tmp.name, "-lm"], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stderr}")
        os.replace(tmp.name, out)
        return out
    finally:
        if os.path.exists(tmp.name):
            os.unlink(tmp.name)


def ensure_built() -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        compile_oracle()
    return LIB


if __name__ == "__main__":
    print(compile_oracle())
