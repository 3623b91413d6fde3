"""Host-side launch logic without a GPU: the dynamic shared-memory opt-in
(``csrc/vn_smem.h``) compiled with the host compiler against stand-ins for the two
CUDA runtime calls it makes (``tests/host/smem_optin.cpp``)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "virtual_noise_perturbed_gb300", "csrc")


def _cuda_include():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    for inc in (os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include"), "/usr/local/cuda/include"):
        if os.path.exists(os.path.join(inc, "cuda_runtime_api.h")):
            return inc
    return None


def test_dynamic_smem_optin_is_per_device_and_thread_safe(tmp_path):
    gxx = shutil.which("g++")
    inc = _cuda_include()
    if gxx is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "smem_optin")
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-Wall", "-I", CSRC, "-I", inc,
                    os.path.join(ROOT, "tests", "host", "smem_optin.cpp"), "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
