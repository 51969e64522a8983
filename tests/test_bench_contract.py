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


def test_device_arm_line_keys_with_the_gpu_run_stubbed(orc_lib, monkeypatch, capsys):
    """The device arm's JSON line, its GPU run replaced by fixed figures: the
    whole-job values, the roofline object, clocks, e2e, the launch count and
    a cpu_baseline from the oracle (rank 0, one GPU)."""
    sys.path.insert(0, ROOT)
    import bench

    fake = {"total_ms": 500.0, "frame_ms": 4.9, "weight_bytes": 1, "bytes_per_frame": 2.0e9, "achieved_gbs": 400.0,
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9},
            "e2e": {"value": 190.0, "s": 0.52, "frames": 100, "h2d": 4096, "d2h": 512},
            "model_device_bytes": 11 << 30}
    monkeypatch.setattr(bench, "run_gpu", lambda *a, **k: fake)
    monkeypatch.setattr(bench, "dist_setup", lambda: (1, 0, 0))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "tiny", "--steps", "100", "--warmup", "3",
                                      "--no-sweep", "--oracle-frames", "1"])
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["value"] == pytest.approx(1 * 100 / 0.5)  # B x steps / seconds
    assert d["ms_per_step"] == pytest.approx(5.0)
    assert (d["n_gpus"], d["steps"], d["warmup"], d["scaling"]) == (1, 100, 3, "weak")
    assert d["unit"] == "frames/s" and d["higher_is_better"] is True and d["vs_baseline"] is None
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] == 400.0
    assert r["frac"] == pytest.approx(400.0 / r["peak"])
    assert r["traffic"] is None  # the traffic record is for full_b1, not tiny
    assert d["e2e"]["value"] == pytest.approx(100 / 0.52)
    assert (d["e2e"]["h2d_bytes_per_step"], d["e2e"]["d2h_bytes_per_step"]) == (4096, 512)
    assert d["gpu_launches"] == 200 and d["clocks"]["sm_mhz"] == 2070.0
    assert d["model_device_bytes"] == 11 << 30
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert d["config"]["workload"].startswith("tiny") and d["config"]["global_batch"] == 1
