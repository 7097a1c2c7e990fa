"""The range-check decisions of the checked build, on the host: tests/native/
checks_host.cpp builds a buffer table and probes accesses at its edges (listed
and unlisted bank and gradient rows, the appended row, the partial sum's
first row, read-only and writable spans, alignment) against chk_decide, the
function the checked kernels call before every access."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_check_decisions_on_the_host(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("needs g++")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("needs the CUDA headers")
    exe = str(tmp_path / "checks_host")
    src = os.path.join(ROOT, "tests", "native", "checks_host.cpp")
    cmd = [cxx, "-std=c++17", "-O1", "-DAR_CHECKED", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "depth_wise_attention_ar_gb300", "csrc"), "-I", cuda_inc,
           src, "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    p = subprocess.run([exe], capture_output=True, text=True)
    print(p.stdout)
    assert p.returncode == 0, p.stdout
    assert p.stdout.strip().splitlines()[-1].endswith(", 0 failed")
