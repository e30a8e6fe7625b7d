"""The bounds-checked build on the GPU (librot_check.so: guard regions after
every workspace slice, filled before and checked after every micro-group).
Each build runs in its own process (tests/check_build_worker.py)."""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from matrix_optimizer_step_rot_gb300 import binding as B
from matrix_optimizer_step_rot_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
WORKER = os.path.join(HERE, "check_build_worker.py")


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return build.build(), build.build(check=True)


def run(lib, *args):
    env = dict(os.environ, ROT_LIB=lib)
    r = subprocess.run([sys.executable, WORKER, *args], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_checked_steps_keep_every_guard_and_match_the_plain_build(libs, tmp_path):
    plain, checked = libs
    run(plain, "steps", str(tmp_path / "plain.npz"))
    run(checked, "steps", str(tmp_path / "checked.npz"))
    a, b = np.load(tmp_path / "plain.npz"), np.load(tmp_path / "checked.npz")
    assert int(a["status"]) == B.ROT_OK
    assert int(b["status"]) == B.ROT_OK  # no guard was touched by any kernel
    for k in a.files:
        if k != "status":
            assert np.array_equal(a[k], b[k]), k  # the layout does not change a result


def test_overwritten_guard_is_reported(libs):
    _, checked = libs
    before, after = (int(x) for x in run(checked, "corrupt").split())
    assert before == B.ROT_OK
    assert after == B.ROT_ECORRUPT
