"""Host-side logic of the library that needs no GPU, built and run on the CPU.

PerDeviceOnce (csrc/dev_once.h) records per device, thread-safely, that a
kernel's shared-memory limit or a symbol's address has been set up; a process
driving several GPUs, or several threads, must neither skip nor repeat that
setup.  The C++ test program exercises it with 16 threads over 8 fake devices.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_76_gb300", "csrc")


def test_per_device_once(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "dev_once_test")
    src = os.path.join(ROOT, "tests", "host", "dev_once_test.cpp")
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC, src, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
