"""The benchmark's JSON line on the CPU: ``bench.py --impl reference`` (the
oracle timed on the host cores, the reference arm) prints exactly one line
carrying every key of the line the GPU arm prints, with consistent values, and
``bench.py`` refuses option combinations it cannot run."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONTRACT_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _bench(*args, env_extra=None):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_complete_line():
    res = _bench("--impl", "reference", "--workload", "tiny_T256_H2", "--steps", "2", "--warmup", "3")
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, res.stdout
    out = json.loads(lines[0])
    assert CONTRACT_KEYS <= set(out), CONTRACT_KEYS - set(out)
    assert out["impl"] == "reference" and out["n_gpus"] == 1 and out["steps"] == 2 and out["warmup"] == 3
    assert out["higher_is_better"] is True and out["scaling"] == "weak" and out["data"] == "synthetic"
    assert out["value"] > 0 and out["ms_per_step"] > 0
    assert out["config"]["workload"] == "tiny_T256_H2" and out["config"]["T"] == 256
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"] and cb["sample"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_bench_refuses_two_entry_points_at_once():
    res = _bench("--split", "--gated-norm", "--steps", "1")
    assert res.returncode != 0 and "separate entry points" in res.stderr
