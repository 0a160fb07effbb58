"""bench.py's reference arm (the oracle timed on the host cores) on CPU: one
JSON line with the contract's keys on rank 0, nothing and exit 0 on the
other ranks."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3", "--batch", "8"]


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert rec["impl"] == "reference" and rec["metric"] == bench.METRIC
    assert rec["value"] > 0 and rec["unit"] == "state-updates/s" and rec["higher_is_better"] is True
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] == 1
    assert rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    assert rec["config"]["workload"].startswith("b256_fp32")


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
