"""Writes tests/golden/causal_tiny_f32.json from the fp64 oracle only.

The pages print no worked numerical example, so this fixture is a regression
record of the oracle itself on the smallest parity workload (B=1, H=1, N=64,
D=M=16, seed 1): it catches any later, unannounced change to the oracle's
arithmetic.  Its correctness comes from the pins in tests/oracle_pins.py, not
from this file.  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from kernelized_causal_attention_gb300.workloads import WORKLOADS, causal_inputs  # noqa: E402


def main():
    w = WORKLOADS["causal_tiny_f32"]
    q, k, v, g = causal_inputs(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed)
    out, den = oracle.causal_fwd(q, k, v, "recurrent")
    dq, dk, dv = oracle.causal_bwd(q, k, v, g, "recurrent")
    rows = [0, 1, 2, 31, 62, 63]
    rec = {
        "source": "fp64 oracle (oracle/oracle.c), recurrent form; regression record",
        "workload": w.name,
        "shape": [w.B, w.H, w.N, w.D, w.M],
        "seed": w.seed,
        "rows": rows,
        "out": out[0, 0, rows].tolist(),
        "den": den[0, 0, rows].tolist(),
        "dq": dq[0, 0, rows].tolist(),
        "dk": dk[0, 0, rows].tolist(),
        "dv": dv[0, 0, rows].tolist(),
        "sums": {"out": float(out.sum()), "dq": float(dq.sum()), "dk": float(dk.sum()),
                 "dv": float(dv.sum())},
    }
    with open(os.path.join(HERE, "causal_tiny_f32.json"), "w") as f:
        json.dump(rec, f, indent=1)


if __name__ == "__main__":
    main()
