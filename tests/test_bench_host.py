"""The benchmark's reference arm and command line, on the host.

``bench.py --impl reference`` times the float64 oracle on the host cores: it
needs no GPU, so its JSON line is checked here key by key.  Under several
ranks only rank 0 works and prints; fewer than three warm-up steps are
refused.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

import bench

_ROOT = Path(__file__).resolve().parents[1]


def _bench(*args, env=None, timeout=300):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, str(_ROOT / "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, env=e, cwd=str(_ROOT))


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["ms_per_step"] > 0 and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the value is the causal-adjusted FLOPs of one 511-token layer per step over the step time
    p = bench.workloads.CONFIGS[bench.WORKLOAD].problem
    assert abs(d["value"] - p.flops() / (d["ms_per_step"] / 1e3) / 1e12) <= 1e-9 * d["value"] + 1e-12


def test_reference_arm_other_ranks_are_silent():
    r = _bench("--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
               env={"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_too_few_warmup_steps_are_refused():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr
