"""The benchmark's reference arm (the float64 oracle on the host cores) prints
one JSON line with the contract's keys, on the GPU arm's metric and config."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] == d["cpu_baseline"]["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["cpu_model"]
    # the GPU arm's config: same workload keys and the default precision mode
    assert d["config"]["precision"] == "3xf16"
    assert "full stack" in d["config"]["workload"]


def test_one_thread_oracle_sample():
    """The CPU baseline's one-thread leg: the oracle sample in a child process
    with BLAS held to one thread (a small sample of the tiny workload here)."""
    sys.path.insert(0, ROOT)
    import bench

    out = bench.oracle_sample_one_thread("tiny", 2, first_step=1)
    assert out is not None
    value, secs = out
    assert value > 0 and secs > 0
    assert bench.cpu_model()
