"""The bench's JSON contract on the CPU: the reference arm (the oracle timed on the
host) prints one line with the keys the driver reads, and the per-step element
count it reports is the workload's definition (pop x weights for the forward, pop x
parameters for the gradients and the dump), as is the dtype it names."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from virtual_noise_perturbed_gb300 import workloads  # noqa: E402


@pytest.mark.parametrize("number", [1, 2, 3, 4, 5])
def test_step_elements(number):
    wl = workloads.make(number)
    weights = sum(l.out_f * l.in_f for l in wl.layers)
    params = weights + sum(l.out_f for l in wl.layers)
    want = {1: wl.pop * (weights + 2 * params), 2: wl.pop * (weights + 2 * params),
            3: wl.pop * (weights + params), 4: wl.pop * params, 5: wl.pop * weights}[number]
    assert bench.step_elements(wl) == want
    # the JSON line's dtype: bf16 only where the forward runs on the tensor cores
    assert bench.compute_dtype(wl) == {1: "f32", 2: "f32", 3: "bf16", 4: "f32", 5: "bf16"}[number]


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny" and d["config"]["noise_elements_per_step"] == 12544
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_bench_refuses_gaussian_on_other_workloads():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny",
                          "--noise", "gaussian"], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "gaussian" in out.stderr
