"""Write tests/golden/small_case_oracle.json from the CPU oracle alone.

The inputs are the small N=2, T=4, d=256 case (partials and residual
~N(0, 1), gamma = 1 + 0.1 N(0, 1), eps = 1e-6, seed 0) drawn with numpy's
PCG64 so the fixture does not depend on a torch version. The outputs are the
oracle's; the fixture guards the oracle against drift between edits and
between hosts (x86-64 and aarch64).

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def main():
    N, T, d, eps = 2, 4, 256, 1e-6
    rng = np.random.default_rng(0)
    parts = [oracle.bf16_from_float64(rng.standard_normal((T, d)).astype(np.float32).astype(np.float64))
             for _ in range(N)]
    res = oracle.bf16_from_float64(rng.standard_normal((T, d)).astype(np.float32).astype(np.float64))
    gamma = oracle.bf16_from_float64((1 + 0.1 * rng.standard_normal(d)).astype(np.float32).astype(np.float64))
    out = oracle.fused_rmsnorm(parts, res, gamma, eps)
    codes, scales, g = oracle.nvfp4_quantize(out["out_norm"])
    hexs = lambda a: np.ascontiguousarray(a).astype(a.dtype.newbyteorder("<")).tobytes().hex()
    doc = {
        "about": "oracle output for the small N=2, T=4, d=256 case; written by make_golden.py",
        "N": N, "T": T, "d": d, "eps": eps,
        "partials": [hexs(p) for p in parts], "residual": hexs(res), "gamma": hexs(gamma),
        "out_residual": hexs(out["out_residual"]), "out_norm": hexs(out["out_norm"]),
        "nvfp4_codes": codes.tobytes().hex(), "nvfp4_scales": scales.tobytes().hex(),
        "nvfp4_global_scale": float(g),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "small_case_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
