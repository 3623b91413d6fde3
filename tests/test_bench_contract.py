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


PK = {"alu_ops": 152 * 64 * 2.07e9, "issue_ops": 152 * 128 * 2.07e9, "hbm_gbs": 6687.8,
      "bf16_tflops": 1945.4, "source": "measured"}


def _k(ms, launches, elements, flops=0.0, hbm_bytes=0.0):
    return {"ms": ms, "launches": launches, "elements": elements, "flops": flops, "hbm_bytes": hbm_bytes}


def test_roofline_reproduces_a_measured_bench_line():
    """The default step's kernel-pass figures of a GB300 run (the policy forward took
    85.2325 us per launch over 1000 launches; the others less): the dominant kernel is the
    forward, bound by the integer ALU pipe at 12 operations per element."""
    el = 1024 * (64 * 256 + 256 * 256 + 256 * 8)             # 85,983,232 per launch
    per_kernel = {
        "linear_mlp": _k(85.23251131176949, 1000, el * 1000, 2.0 * el * 1000, 632864 * 1000),
        "grad": _k(80.3, 1000, 1024 * 84488 * 1000),
        "noise_dump": _k(80.2, 1000, 1024 * 84488 * 1000, hbm_bytes=4 * 1024 * 84488 * 1000),
        "es_ranks": _k(6.3, 1000, 0),
    }
    r = bench.roofline_of(per_kernel, PK, "no-such-workload")
    assert r["kernel"] == "linear_mlp" and r["bound"] == "alu" and r["unit"] == "Tops/s"
    assert abs(r["achieved"] - 12.105694976249307) < 1e-9
    assert abs(r["frac"] - 0.6011679506861666) < 1e-12
    assert abs(r["issue_frac"] - 0.5260219568503957) < 1e-12
    assert r["peak"] == PK["alu_ops"] / 1e12 and r["ops_per_element"] == 12
    assert r["traffic"] is None and r["launches"] == 1000 and abs(r["avg_launch_us"] - 85.2325113) < 1e-6


def test_roofline_picks_the_tightest_bound():
    n = 10 ** 9
    # a dump whose stores outrun its hashing: HBM binds (4 B per element at 6.6 TB/s
    # against 12 ALU operations per element at 20.1 Tops/s)
    r = bench.roofline_of({"noise_dump": _k(1.0, 1, n, hbm_bytes=4 * n)}, PK, "x")
    assert r["bound"] == "hbm" and abs(r["achieved"] - 4000.0) < 1e-9 and r["unit"] == "GB/s"
    # the Gaussian kind: 32 instructions through a 128-lane issue port bind before 13 ALU
    # operations on the 64-lane pipe or 3 MUFU operations on the 32-lane one
    r = bench.roofline_of({"grad_gaussian": _k(1.0, 1, n)}, PK, "x")
    assert r["bound"] == "issue" and r["ops_per_element"] == 32
    assert abs(r["frac"] - n * 32 / 1e-3 / PK["issue_ops"]) < 1e-12
    # a contraction with few elements and many flops: the tensor pipe binds
    r = bench.roofline_of({"linear_tc": _k(1.0, 1, 10 ** 6, flops=1.5e12)}, PK, "x")
    assert r["bound"] == "tensor" and abs(r["achieved"] - 1500.0) < 1e-9


def test_summary_of_a_measured_workload():
    """summarise(): value from the step pass over the max-over-ranks time, the dominant
    kernel's roofline, shares and the phase metrics from the kernel pass."""
    wl = workloads.make(3)
    el_fwd = 4096 * 1024 * 1024
    per_kernel = {"linear_tc": _k(41.3, 10, el_fwd * 10, 2.0 * el_fwd * 32 * 10),
                  "grad": _k(33.6, 20, 4096 * (1024 * 1024 + 1024) * 10)}
    per_kernel["grad"]["grad_w_elems"] = 1024 * 1024 * 10
    per_kernel["linear_tc"]["grad_w_elems"] = 0
    res = {"per_kernel": per_kernel, "el_step": bench.step_elements(wl), "steps": 10, "total_ms_max": 75.0,
           "graph": True, "graph_error": None}
    s = bench.summarise(wl, res, 1, PK)
    assert abs(s["value"] - bench.step_elements(wl) * 10 / 75e-3) < 1.0
    assert abs(s["ms_per_step"] - 7.5) < 1e-12 and s["steps"] == 10
    assert s["roofline"]["kernel"] == "linear_tc" and s["roofline"]["bound"] == "alu"
    assert abs(sum(k["share"] for k in s["kernels"].values()) - 1.0) < 1e-12
    assert abs(s["perturbed_linear_tflops"] - 2.0 * el_fwd * 32 * 10 / 41.3e-3 / 1e12) < 1e-9
    assert abs(s["grad_w_elem_per_s"] - 1024 * 1024 * 10 / 33.6e-3) < 1e-3
    assert "CUDA graph" in s["launch"]


def test_measured_ceiling_sits_beside_the_derived_peak():
    r = bench.roofline_of({"grad": _k(1.0, 1, 10 ** 9)}, PK, "x")
    hp = {"tops": 16.4}
    bench.with_measured_peak(r, hp)
    assert r["peak"] == PK["alu_ops"] / 1e12                       # the derived peak stays the peak
    assert r["peak_measured"] == 16.4 and abs(r["frac_of_measured"] - r["achieved"] / 16.4) < 1e-12
    h = bench.roofline_of({"noise_dump": _k(1.0, 1, 10 ** 9, hbm_bytes=4e9)}, PK, "x")
    bench.with_measured_peak(h, hp)
    assert "peak_measured" not in h                                 # only alu-bound rooflines
    bench.with_measured_peak(r, None)                               # no probe run: unchanged


def test_default_extras_and_refusals():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--extras", "mid,nope"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "nope" in out.stderr
    assert bench.EXTRA_DEFAULT == ["mid", "grad_only", "es_mlp", "tiny"]
