"""Write tests/golden/tiny_oracle.json: oracle values for the tiny workload.

Calls only the float64 oracle and the seeded input generator.  The tiny
workload is the README "Usage / AscendC inference" demo shape
[1,128,2,64,128,128,1] (fp32, dt_softplus, final state returned).
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import ssd_inputs  # noqa: E402


def main():
    w = ssd_inputs.WORKLOADS["tiny"]
    inp = ssd_inputs.make(w)
    prob = oracle.Problem(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                          dt_softplus=inp["dt_softplus"])
    y, fin = oracle.forward(prob)
    picks = [(0, 0, 0, 0), (0, 0, 1, 5), (0, 17, 0, 63), (0, 64, 1, 31), (0, 127, 1, 0),
             (0, 127, 0, 40)]
    fpicks = [(0, 0, 0, 0), (0, 1, 63, 127), (0, 0, 10, 100), (0, 1, 32, 7)]
    out = {
        "_source": "float64 oracle on ssd_inputs.WORKLOADS['tiny'] (seed 1); written by tests/golden/make_golden.py",
        "y_samples": [[list(p), float(y[p])] for p in picks],
        "final_samples": [[list(p), float(fin[p])] for p in fpicks],
        "y_l2": float(np.linalg.norm(y.ravel())),
        "final_l2": float(np.linalg.norm(fin.ravel())),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
