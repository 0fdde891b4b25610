"""Failure detection without a GPU fault.

The library's kernels never trap: every wait on an mbarrier is bounded (1 s of
%globaltimer), after which the kernel ORs EP_ERRF_TIMEOUT into the caller's
flag word and returns.  Here that wait is made to run out on purpose -- an
mbarrier armed for bytes that no copy delivers -- and the test checks that
the flag arrives, that the wait lasted about the bound, and that the context
still runs a real bulk copy and a plain kernel afterwards.  Bad arguments are
refused on the host (tests/test_abi.py); bad ids, capacity drops and bad slots
are flagged on the device (tests/test_gpu_parity.py).
"""
import os
import re
import subprocess

import pytest

import combine_ep_get_04_gb300 as ep

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "combine_ep_get_04_gb300", "csrc")

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_and_leaves_the_context_usable(tmp_path):
    from combine_ep_get_04_gb300 import build as B
    exe = tmp_path / "wait_timeout"
    subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-std=c++17", "--expt-relaxed-constexpr", "-I", CSRC,
                    os.path.join(HERE, "wait_timeout.cu"), "-o", str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout
    f = dict(kv.split("=", 1) for kv in out.split())
    assert int(f["timeout_flag"]) == int(f["timeout_bit"]) == ep.ERRF_TIMEOUT, out
    assert 900.0 <= float(f["waited_ms"]) <= 1500.0, out
    assert f["err1"] == f["err2"] == f["err3"] == "cudaSuccess", out
    assert int(f["delivered_flag"]) == 0 and f["delivered_ok"] == "1", out
    assert f["plain_ok"] == "1", out
