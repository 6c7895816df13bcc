"""bench.py's reference arm (the oracle on the host cores), on CPU.

Rank 0 alone runs the oracle and prints one JSON line; under a multi-rank
launch every other rank exits 0 without work or output.
"""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_rank0_prints_one_reference_line():
    r = _run({"RANK": "0"})
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    assert out["value"] > 0 and out["higher_is_better"] is True
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["value"] == out["value"]
    assert out["cpu_baseline"]["cores"] >= 1
    assert out["e2e"] == {"value": out["value"], "unit": out["unit"],
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert out["config"]["workload"].startswith("tiny:")


def test_other_ranks_exit_without_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
