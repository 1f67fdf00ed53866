"""The benchmark's JSON contract on the paths that need no GPU: the reference
arm (the fp64 oracle timed on host cores) and the oracle child process that
the GPU arm uses for its CPU baseline."""

from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _last_json(cmd, env=None):
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, **(env or {})))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_line():
    line = _last_json([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                       "--warmup", "1"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["dtype"] == "f64" and line["data"] == "synthetic"
    cfg = line["config"]
    assert cfg["S"] == 256 and cfg["Hq"] == 32 and cfg["Hkv"] == 8 and cfg["D"] == 128
    assert cfg["kv_bytes_per_step"] == cfg["context_tokens"] * 2 * 8 * 128 * 2
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_oracle_child_line():
    # the child that times the oracle for the GPU arm's cpu_baseline: whole
    # batch on one thread, then one process per core
    line = _last_json([sys.executable, "bench.py", "--_oracle-sample", "tiny"],
                      env={"OMP_NUM_THREADS": "1"})
    assert line["kind"] == "oracle" and line["cores"] == 1 and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["seconds"] > 0
    assert "4 sequences" in line["sample"]
    if "all_cores" in line:
        assert line["all_cores"]["cores"] >= 2 and line["all_cores"]["value"] > 0
