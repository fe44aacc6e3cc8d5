"""Writes tests/golden/loftq_4096_r16_T5.json from the CPU oracle only.

Input: the LoftQ workload of the seeded generators (4096 x 4096 fp32,
Student-t with 4 degrees of freedom scaled to std 0.02, seed 4); r = 16,
alpha = 16, T = 5, NF4 with double quantisation.  The file records the
residuals ||W - deq(Q_t) - s B_t A_t||_F for t = 0..5 computed with the exact
LAPACK SVD of the oracle.  Run from the repository root:

    python tests/golden/make_loftq_golden.py
"""

import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import loftq  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "loftq_4096_r16_T5.json")


def main():
    t0 = time.time()
    W = synth.loftq_case(seed=4, d=4096, k=4096)
    res = loftq.loftq(W, r=16, alpha=16.0, T=5)
    out = {
        "workload": "LoftQ 4096x4096 fp32 Student-t(df=4) std 0.02, seed 4; r=16, alpha=16, T=5, NF4+DQ",
        "source": "oracle.loftq.loftq (float64, numpy.linalg.svd)",
        "resid": res.resid,
        "seconds": time.time() - t0,
    }
    with open(OUT, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
