"""The fp8 quantiser divides through a corrected reciprocal instead of an
IEEE division (Markstein's quotient correction); the block scale and every
e4m3 code must stay exactly those of the IEEE quotient.

CPU: the method itself in plain C against C's IEEE division over the inputs a
quantiser sees.  GPU: the library's device code (ep_device.cuh) against
CUDA's __fdiv_rn for every bf16 amax and every bf16 x a block with that
amax can hold, for f32 and UE8M0 scales.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "combine_ep_get_04_gb300", "csrc")


def test_quotient_correction_matches_ieee_division_in_c(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "quotient_method"
    subprocess.run([gcc, "-std=c11", "-O2", "-ffp-contract=off", os.path.join(HERE, "quotient_method.c"), "-o",
                    str(exe), "-lm"], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=300).stdout
    m = re.search(r"pairs=(\d+) mismatches=(\d+)", out)
    assert m, out
    assert int(m.group(1)) > 14_000_000
    assert int(m.group(2)) == 0, out


@pytest.mark.gpu
def test_quantiser_quotients_match_fdiv_exhaustively(tmp_path):
    from combine_ep_get_04_gb300 import build as B
    exe = tmp_path / "quotient_exhaustive"
    subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-std=c++17", "--expt-relaxed-constexpr", "-I", CSRC,
                    os.path.join(HERE, "quotient_exhaustive.cu"), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=300).stdout
    lines = [l for l in out.splitlines() if l.startswith("ue8m0=")]
    assert len(lines) == 2, out
    for line in lines:
        f = dict(kv.split("=") for kv in line.split())
        assert int(f["pairs"]) > 2_000_000_000, line
        # the quantiser's domain: |x| <= amax of the block (code_mismatch_out
        # counts |x| > amax, which no block holds, and is reported only)
        for key in ("scale_mismatch", "code_mismatch_in", "quotient_mismatch_in"):
            assert int(f[key]) == 0, line
    assert "cuda=no error" in out
