"""Writes oracle_regression.json: the float64 oracle's results on a small
seeded case, stored as exact hexadecimal floats.  Calls only the oracle and
the seeded input generator.  The file freezes the oracle's outputs: any later
change to its arithmetic shows up as a mismatch in tests/test_golden.py.

    python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from matrix_optimizer_step_rot_gb300 import inputs  # noqa: E402
from oracle import rot_oracle as orc  # noqa: E402

SHAPES = ((6, 4), (4, 6), (5, 5))
STEPS, K = 4, 2


def workload():
    return inputs.Workload("golden", SHAPES, ("a", "b", "c"), 0.02, 1e-2, "normal", STEPS, K,
                           1 << 20, 7)


def compute():
    wl = workload()
    out = {"shapes": SHAPES, "steps": STEPS, "refresh_every": K, "seed": 7, "matrices": []}
    for i, (W, st) in orc.run(wl).items():
        out["matrices"].append({
            "index": i,
            "W": [float(x).hex() for x in W.ravel()],
            "U": [float(x).hex() for x in st.U.ravel()],
            "V": [float(x).hex() for x in st.V.ravel()],
            "rank_u": int(st.rank_u), "rank_v": int(st.rank_v),
        })
    plan = orc.plan(SHAPES, c_max=200, ranks=2)
    out["plan"] = {"c_max": 200, "ranks": 2, "groups": plan.groups, "owners": plan.owners}
    part = orc.alpha_partition([orc.item_cost(m, n) for m, n in SHAPES], [2, 1], 2, 1.0)
    out["alpha_partition"] = {"buckets": [2, 1], "ranks": 2, "alpha": 1.0,
                              "owners": part.owners, "loads": part.loads}
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(compute(), f, indent=1)
