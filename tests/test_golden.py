"""The oracle against its stored results (tests/golden/oracle_regression.json,
written by tests/golden/make_golden.py from the oracle itself).  Plans and
partitions must match exactly; floating-point results to 1e-10 relative, which
allows for BLAS and compiler rounding differences between machines but not for
a change to the arithmetic."""

import json
import os

import numpy as np

from tests.golden import make_golden as G
from oracle import rot_oracle as orc

HERE = os.path.dirname(os.path.abspath(__file__))


def load():
    with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
        return json.load(f)


def unhex(xs, shape):
    return np.array([float.fromhex(x) for x in xs]).reshape(shape)


def test_oracle_reproduces_stored_results():
    stored = load()
    got = G.compute()
    assert got["plan"] == stored["plan"]
    assert got["alpha_partition"] == stored["alpha_partition"]
    for a, b in zip(got["matrices"], stored["matrices"]):
        m, n = stored["shapes"][b["index"]]
        assert (a["rank_u"], a["rank_v"]) == (b["rank_u"], b["rank_v"])
        for key, shape in (("W", (m, n)), ("U", (m, m)), ("V", (n, n))):
            x, y = unhex(a[key], shape), unhex(b[key], shape)
            assert np.linalg.norm(x - y) <= 1e-10 * np.linalg.norm(y), key
