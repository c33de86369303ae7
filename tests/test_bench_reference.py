"""The benchmark's reference arm (the CPU oracle on a bounded sample), on CPU:
one JSON line with the contract's keys from rank 0, nothing from other ranks,
and a per-step sample that shrinks as the step count grows."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_line_has_the_contract_keys():
    r = _run("--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert "16 of 16 units" in line["config"]["sample"]  # a few steps: the whole sample each step


def test_reference_other_ranks_print_nothing():
    r = _run("--steps", "2", "--warmup", "1", env={"RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_sample_shrinks_with_many_steps():
    """The whole sample for a few steps; one or two units per step at the
    default 1000 steps (plus warm-up), one when a unit alone is slow."""
    import bench
    assert bench.units_per_step(0.06, 4, 16) == 16
    assert bench.units_per_step(0.06, 1005, 16) in (1, 2)
    assert bench.units_per_step(0.06, 1005, 16) * 1005 * 0.06 <= bench.REFERENCE_BUDGET_S
    assert bench.units_per_step(10.0, 1005, 16) == 1
    assert bench.units_per_step(0.06, 0, 16) == 16
