"""Writes small_case.json: a small seeded case and the oracle's outputs for it.

The stored values come from the CPU oracle only (this script imports nothing
else that computes the decode). It is a regression fixture: a later change to
the oracle's arithmetic that moves these values must say why.

    python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from sparse_mla_decode_gb300 import inputs  # noqa: E402


def main():
    case = inputs.random_case(77, B=3, H=16, W=12, N=20, counts=[12, 0, 5], heavy_frac=0.1)
    out, _, lse = oracle.sparse_mla_decode(case.q8, case.kv8, case.indices, case.counts,
                                           case.sm_scale, case.q_scale, case.k_scale)
    g = {
        "what": "sparse MLA decode, B=3 H=16 W=12 N=20 counts [12,0,5]; outputs from the oracle",
        "B": case.B, "H": case.H, "W": case.W, "N": case.N,
        "sm_scale": case.sm_scale, "q_scale": case.q_scale, "k_scale": case.k_scale,
        "q8": case.q8.tobytes().hex(), "kv8": case.kv8.tobytes().hex(),
        "indices": case.indices.reshape(-1).tolist(), "counts": case.counts.tolist(),
        "out_bf16": out.reshape(-1).tolist(),
        "lse": [None if math.isinf(v) else float(v) for v in lse.reshape(-1)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "small_case.json")
    with open(path, "w") as f:
        json.dump(g, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
