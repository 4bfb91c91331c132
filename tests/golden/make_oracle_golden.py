"""Write oracle_small_case.json: the oracle's own output on a small seeded case.

It calls only the oracle and the input generator.  The stored values let the
test suite check that the oracle gives bit-identical results on every machine
it runs on (x86 and Arm hosts).  Run from the repository root:

    python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import oracle as o  # noqa: E402
from sparse_attention_paged_dsa_gb300 import inputs as I  # noqa: E402

CASE = dict(name="golden", batch=3, max_context=1024, seq_lens=[300, 9, 1024], num_pages=12,
            k=40, seed=4242)


def main():
    c = I.make_case(**CASE)
    s = o.case_scores(c)
    t = o.case_topk(c, s)
    out = {
        "note": "written by tests/golden/make_oracle_golden.py from the oracle alone",
        "case": CASE,
        "live_scores_hex": [float.hex(float(x)) for x in s[np.isfinite(s)]],
        "topk": t.tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_case.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=0)
        f.write("\n")


if __name__ == "__main__":
    main()
