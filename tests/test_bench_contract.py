"""The benchmark's reference arm keeps the output contract on the host alone (CPU only): one
JSON line with the metric, the value, the timing and configuration keys, the CPU-baseline
description and the end-to-end object, for an fp64 and an INT8 workload; non-zero ranks of a
multi-rank launch print nothing."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
        "e2e"}


def run_reference(workload, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--workload", workload],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.strip()]


@pytest.mark.parametrize("workload,dtype", [("tiny_dwpw_f32", "f64"), ("pwpw_i8", "int8")])
def test_reference_arm_line(workload, dtype):
    lines = run_reference(workload)
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["dtype"] == dtype and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    assert d["config"]["workload"] == workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    assert run_reference("tiny_dwpw_f32", {"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_gpu_arm_fails_loudly_without_a_gpu():
    """No CPU fallback: without a GPU the measured arm exits non-zero and prints no result."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1", "--warmup",
                        "1", "--no-cpu-baseline"], capture_output=True, text=True, cwd=ROOT,
                       timeout=600)
    assert r.returncode != 0
    assert not any(l.startswith("{") for l in r.stdout.splitlines())
