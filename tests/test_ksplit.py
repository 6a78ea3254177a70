"""Host-only test of the tensor-core GEMM's K-split choice: builds
tests/ksplit_test.cc against decoder_only_forward_gb300/csrc/ksplit.h with the
host C++ compiler and runs it.  No GPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_ksplit_choice(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "ksplit_test")
    src = os.path.join(ROOT, "tests", "ksplit_test.cc")
    inc = os.path.join(ROOT, "decoder_only_forward_gb300", "csrc")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-I", inc, src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ksplit ok" in r.stdout
