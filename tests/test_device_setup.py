"""Host-side check of the per-device launch set-up, on the CPU.

The dynamic shared-memory limit and the resident-CTA count of a kernel belong
to one device; the library keys both by (device, kernel) behind one mutex.  This
test compiles the library's device_setup.cpp against a fake CUDA runtime
(tests/fake_cudart_setup.cpp) whose current device the test switches, and checks
that every device is configured once, that resident CTAs follow each device's
SM count, and that concurrent host threads configure a device once.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = "/usr/local/cuda/include"


def test_per_device_launch_setup(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INCLUDE, "cuda_runtime_api.h")):
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / "device_setup_check"
    csrc = os.path.join(ROOT, "kv_buffered_decoding_gb300", "csrc")
    cmd = [gxx, "-std=c++17", "-O1", "-pthread",
           "-I", os.path.join(ROOT, "include"), "-I", csrc, "-I", CUDA_INCLUDE,
           os.path.join(csrc, "device_setup.cpp"),
           os.path.join(ROOT, "tests", "fake_cudart_setup.cpp"),
           "-o", str(exe)]
    build = subprocess.run(cmd, capture_output=True, text=True, timeout=240)
    assert build.returncode == 0, build.stderr[-2000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip().endswith("ok"), run.stdout + run.stderr
