"""The work-map arithmetic the kernels share with the host, checked on the
CPU: tests/native/host_logic.cpp includes the library's internal header and
tests the per-expert tile plan, the tile-list bound the workspace and the
checked builds rely on, the checked builds' tile-entry test and the MXFP8
per-tile scale layout."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_logic(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if not cxx or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    exe = tmp_path / "host_logic"
    src = os.path.join(ROOT, "tests", "native", "host_logic.cpp")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-I", os.path.join(cuda, "include"),
                        src, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout
