"""Write the oracle golden fixtures in this folder.

Calls only ``oracle`` (the fp64 CPU oracle) and ``workloads`` (seeded input
generators); nothing here touches the CUDA library.  Re-run it only when the
definition or a generator recipe changes on purpose, and say why in the commit.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def main() -> None:
    o = oracle.default()
    cases = {}
    for inp in (W.tiny(), W.sweep(8, 2048, z=0.0), W.decode(4)):
        bits = W.to_bits(inp.x)
        res = o.gelu_and_mul_sparse(bits, d=inp.d, z=inp.z)
        ref16 = np.array([o.double_to_bf16(v) for v in res.ref.ravel()], dtype=np.uint16)
        cases[inp.name] = {
            "T": inp.T, "d": inp.d, "row_stride": inp.row_stride, "z": inp.z, "seed": inp.seed,
            "input_sha256": digest(bits),
            "row_mean": res.mean.tolist(), "row_std": res.std.tolist(),
            "row_cutoff": res.cutoff.tolist(),
            "nonzero_count": int((res.ref != 0).sum()),
            "ref_sum": float(res.ref.sum()), "ref_abs_sum": float(np.abs(res.ref).sum()),
            "ref_bf16_sha256": digest(ref16),
        }
    s = W.silu(1024)
    r64, r16 = o.silu_and_mul(W.to_bits(s))
    cases["silu_M1024"] = {"M": 1024, "d": W.SILU_D, "seed": 3 + 1024,
                           "input_sha256": digest(W.to_bits(s)),
                           "ref_sum": float(r64.sum()), "ref_bf16_sha256": digest(r16)}
    out = {"generated_by": "tests/golden/make_golden.py (oracle + workloads only)",
           "torch_version": torch.__version__, "cases": cases}
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
