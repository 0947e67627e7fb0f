"""Write tests/golden/tiny_rows.json: oracle outputs on sampled rows of the tiny
workload (1 x 256 x 1 head, d = 64, non-causal, seed 1001).

Calls only the fp64 oracle (oracle/) and the seeded input generator.  Run from the
repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle.oracle as ORACLE  # noqa: E402
from exact_attention_81_gb300.inputs import WORKLOADS, workload_inputs  # noqa: E402

ROWS = [0, 1, 2, 63, 64, 127, 128, 200, 254, 255]


def main():
    w = WORKLOADS["tiny"]
    q, k, v = workload_inputs(w)
    rows = np.array([[0, 0, i] for i in ROWS], np.int32)
    o, lse = ORACLE.attention_rows(q, k, v, rows, w.scale, w.causal)
    out = {
        "what": "fp64 oracle on rows of the tiny workload: B=1, H=1, N=256, d=64, "
                "non-causal, scale=1/8, bf16 iid N(0,1) from seed 1001 "
                "(exact_attention_81_gb300.inputs.dense_inputs)",
        "written_by": "tests/golden/make_golden.py (oracle only)",
        "rows": ROWS,
        "o": [[float(x) for x in r] for r in o],
        "lse": [float(x) for x in lse],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_rows.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
