"""The benchmark's JSON line, checked on the CPU through its reference arm
(the fp64 oracle timed on the host cores), and its GPU arm's refusal to run
without a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_json_line():
    r = _bench("--impl", "reference", "--steps", "2", "--warmup", "1", "--shape", "64,256,128")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["dtype"] == "f64" and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "1", "--shape", "64,256,128",
               env_extra={"RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_gpu_arm_fails_loudly_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the GPU arm would run")
    r = _bench("--steps", "1", "--warmup", "3", "--e2e-steps", "0", "--no-cpu-baseline", "--no-context")
    assert r.returncode != 0
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_compact_headline_keeps_the_rates_and_fractions():
    """The stdout line's headline block: per shape the times, the rate and both
    fractions; the full record keeps the rest."""
    sys.path.insert(0, ROOT)
    import bench
    full = {"4096x4096x4096 bf16": {"us": 74.86, "us_single_calls": 86.64, "copies": 7, "tile": "256x256",
                                    "TFLOP/s": 1836.0, "of_nominal": 0.816, "of_measured": 0.952,
                                    "target_of_nominal": 0.7},
            "16x4096x4096 bf16": {"us": 8.82, "us_single_calls": 9.49, "copies": 13, "tile": "decode",
                                  "GB/s": 3832.9, "of_nominal": 0.4791, "of_measured": 0.5734,
                                  "target_of_nominal": 0.6}}
    got = bench.compact_headline(full)
    assert got == {"4096x4096x4096 bf16": {"us": 74.86, "us_single_calls": 86.64, "TFLOP/s": 1836.0,
                                           "of_nominal": 0.816, "of_measured": 0.952},
                   "16x4096x4096 bf16": {"us": 8.82, "us_single_calls": 9.49, "GB/s": 3832.9,
                                         "of_nominal": 0.4791, "of_measured": 0.5734}}
    assert bench.compact_headline(None) is None
