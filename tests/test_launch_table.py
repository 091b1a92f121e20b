"""The per-device launch bookkeeping (csrc/launch_table.h: the shared-memory
opt-in done once per (device, kernel), the occupancy cache) on the host: a
C++ check with made-up devices and a fake attribute setter, compiled with the
host compiler and run here.  No GPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_launch_tables_two_devices_and_racing_threads():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "launch_table_check")
        subprocess.run([cxx, "-std=c++17", "-O1", "-pthread",
                        "-I", os.path.join(ROOT, "swiglu_mlp_group_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "launch_table_check.cc"), "-o", exe],
                       check=True, capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
        assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
