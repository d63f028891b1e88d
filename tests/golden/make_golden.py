"""Writes tests/golden/oracle_small.json: small inputs and the fp64 oracle's outputs.

The pages print no worked example for this method, so these fixtures are the
oracle's own values on a few small seeded inputs: they freeze the oracle so that
a later change to its arithmetic shows up in tests/test_golden.py. The script
calls only ``oracle`` (and the seeded input generator for the inputs).

Run from the repository root: ``python tests/golden/make_golden.py``.
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from tiled_newton_schulz_03_b300 import synth  # noqa: E402

CASES = [
    # name, H, W, T, K, coeffs, norm, generator
    ("gauss_6x10_T4_K3", 6, 10, 4, 3, oracle.QUINTIC, "tile", "gaussian"),
    ("lowrank_9x7_T8_K5", 9, 7, 8, 5, oracle.QUINTIC, "tile", "lowrank"),
    ("gauss_5x5_T5_K2_cubic", 5, 5, 5, 2, (1.5, -0.5, 0.0), "tile", "gaussian"),
    ("gauss_7x12_T4_K1_matrix", 7, 12, 4, 1, oracle.QUINTIC, "matrix", "gaussian"),
]


def main():
    out = []
    for i, (name, H, W, T, K, coeffs, norm, gen) in enumerate(CASES):
        if gen == "gaussian":
            G = synth.gaussian(H, W, seed=1000 + i).double().numpy()
        else:
            G = synth.lowrank_noise(H, W, seed=1000 + i, rank=2, scale=1.0,
                                    noise_std=0.1).double().numpy()
        O = oracle.tiled_ns(G, T, K, coeffs, norm, oracle.DEFAULT_EPS)
        out.append({"name": name, "H": H, "W": W, "T": T, "K": K,
                    "coeffs": list(coeffs), "norm": norm, "eps": oracle.DEFAULT_EPS,
                    "input": [repr(float(v)) for v in G.ravel()],
                    "output": [repr(float(v)) for v in O.ravel()]})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as f:
        json.dump({"source": "fp64 oracle (oracle/himuon_oracle.py); written by "
                             "tests/golden/make_golden.py", "cases": out}, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
