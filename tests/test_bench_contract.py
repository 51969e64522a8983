"""The bench's reference arm (the oracle on the host cores) keeps the JSON-line
contract: one line on stdout with the metric, its unit and direction, the run
shape, the workload, a cpu_baseline describing the run and an end-to-end
figure with no host-device copies; ranks other than 0 of a multi-GPU launch
print nothing and exit 0."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(args, env_extra=None, timeout=600):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          cwd=ROOT, env=env, timeout=timeout)


@pytest.fixture(scope="module")
def ref_line(orc_lib):
    r = run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_line_keys(ref_line):
    d = ref_line
    assert d["impl"] == "reference"
    assert d["metric"].startswith("codec frames/s")
    assert d["unit"] == "frames/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["config"]["workload"].startswith("tiny")


def test_reference_cpu_baseline_and_e2e(ref_line):
    d = ref_line
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and "tiny" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_other_ranks_are_silent(orc_lib):
    r = run_bench(["--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3"],
                  {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
