"""The bf16 dispatch ring's load schedule, checked on the CPU: after a wait
gives up, the kernel drains exactly the loads still in flight (none may land
in shared memory after the CTA exits), and no stage is reloaded before the
unit that used it was waited for."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "combine_ep_get_04_gb300", "csrc")


def test_ring_schedule_drains_every_load_in_flight(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "ring_schedule_check"
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(HERE, "ring_schedule_check.cpp"), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "ring schedule ok" in res.stdout
