"""Write tests/golden/oracle_cases.json: expected results of the CPU oracle on
seeded uniform inputs in the shapes of the five workloads (and a few odd
sizes), for the regression tests of the oracle (tests/test_golden.py) and the
library (tests/test_gpu_golden.py).

Every stored value comes from oracle/ alone; the inputs come from synth's
integer-only uniform generators, so both sides rebuild them exactly from the
stored seed and shape.  Run from the repository root:

    python -m tests.golden.make_oracle_golden

A change of a stored value must name, in its commit message, the passage (or
the reading of it) that justifies the oracle change behind it.
"""
from __future__ import annotations

import json
import os

import oracle
from tests.golden import case_inputs

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_cases.json")

# kind, seed, n, w, h, bpc -- the shapes of the five workloads and odd sizes
CASES = [
    ("motion", 101, 2, 64, 48, 8),          # the 64x48 pair
    ("motion", 102, 6, 576, 324, 8),        # the 576x324 sequence (first frames)
    ("motion", 103, 3, 1920, 1080, 8),      # the 1080p sequence (first frames)
    ("motion", 105, 2, 3840, 2160, 10),     # the 4K 10-bit sequence (first frames)
    ("motion", 109, 4, 67, 35, 16),         # odd size, 16 bits
    ("motion", 110, 4, 130, 34, 12),        # one tile and a ragged column, 12 bits
    ("motion_v2", 106, 4, 576, 324, 8),
    ("motion_v2", 107, 4, 130, 34, 10),
    ("motion_v2", 111, 3, 67, 35, 16),
    ("yuv420", 104, 2, 3840, 2160, 8),      # the 4K 4:2:0 pairs (first pairs)
    ("yuv420", 112, 3, 257, 70, 10),        # odd size, 10 bits
    ("moments", 108, 2, 576, 324, 8),
    ("moments", 113, 2, 67, 35, 16),
]


def expected(o: oracle.Oracle, kind: str, data, bpc: int) -> dict:
    if kind == "motion":
        return {"sad": [int(v) for v in o.motion_sad_sequence(data, bpc)]}
    if kind == "motion_v2":
        return {"sad": [int(v) for v in o.motion_v2_sequence(data, bpc)]}
    if kind == "yuv420":
        sse = [[int(o.sse(data.ref_y[i], data.dist_y[i], bpc)), int(o.sse(data.ref_u[i], data.dist_u[i], bpc)),
                int(o.sse(data.ref_v[i], data.dist_v[i], bpc))] for i in range(data.n)]
        return {"sad": [int(v) for v in o.motion_sad_sequence(data.ref_y, bpc)], "sse": sse}
    return {"sums": [[int(v) for v in o.moment_sums(data.ref_y[i], data.dist_y[i], bpc)]
                     for i in range(data.n)]}


def main() -> None:
    o = oracle.Oracle()
    cases = []
    for kind, seed, n, w, h, bpc in CASES:
        data = case_inputs(kind, seed, n, w, h, bpc)
        cases.append({"kind": kind, "seed": seed, "n": n, "w": w, "h": h, "bpc": bpc,
                      **expected(o, kind, data, bpc)})
    doc = {"source": "written by tests/golden/make_oracle_golden.py from oracle/ alone; inputs are "
                     "synth.uniform_frames / synth.uniform_yuv420 with the stored seed and shape",
           "cases": cases}
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
