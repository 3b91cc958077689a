"""Writes tests/golden/tiny_oracle_samples.json.

Calls only the oracle (and the seeded input generator for its inputs): the
stored values are the fp64 oracle's outputs on the tiny workload (B=1, T=64,
H_qk=2, H_v=4, d=32, fp32, chunk 16, seed 0), kept as a regression guard for
the oracle and the generator.  Re-run only when one of them changes on purpose:

    python tests/golden/make_oracle_samples.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from gated_deltanet_scan_gb300 import synth  # noqa: E402

SAMPLES = [(0, 0, 0), (5, 1, 7), (15, 2, 31), (16, 3, 0), (33, 0, 12), (63, 3, 31), (63, 1, 5)]


def main():
    w = synth.tiny()
    o, S = oracle.run_workload(w, threads=1)
    out = {
        "_about": "fp64 oracle on the tiny workload (seed 0); written by make_oracle_samples.py",
        "inputs_checksum": {
            "q_sum": float(np.sum(w.q, dtype=np.float64)),
            "v_sum": float(np.sum(w.v, dtype=np.float64)),
            "g_sum": float(np.sum(w.g, dtype=np.float64)),
            "beta_sum": float(np.sum(w.beta, dtype=np.float64)),
        },
        "o_samples": [[t, h, j, float(o[t, h, j])] for (t, h, j) in SAMPLES],
        "o_rms": float(np.sqrt(np.mean(o * o))),
        "state_fro": [float(np.linalg.norm(S[0, h])) for h in range(w.h_v)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_samples.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
