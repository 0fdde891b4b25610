"""The pins catch plausible mistakes in the oracle.

Each case compiles a copy of the oracle's C source with one planted mistake
(a dropped term, a wrong index, a reversed order, a wrong rounding rule; all
of them stay inside the buffers) into a temporary library, points the oracle
wrapper at it in a fresh Python process, and checks that at least one of the
pin checks fails.  Nothing here touches a GPU or the product path.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.c")

MUTATIONS = {
    "combine drops a term": ("bf16_bits_to_f32(y[slot * H + i]);\n                acc = acc + prod;",
                             "bf16_bits_to_f32(y[slot * H + i]);\n                acc = prod;"),
    "combine wrong weight index": ("topk_w[(long)t * k + j] * bf16", "topk_w[(long)t * k] * bf16"),
    "combine wrong row": ("bf16_bits_to_f32(y[slot * H + i])", "bf16_bits_to_f32(y[(long)t * H + i])"),
    "layout reversed order in expert": ("slot = offsets[e] + rank;", "slot = offsets[e + 1] - 1 - rank;"),
    "layout walks j before t": ("for (int t = 0; t < T; ++t) {\n        for (int j = 0; j < k; ++j) {\n            long n",
                                "for (int j = 0; j < k; ++j) {\n        for (int t = 0; t < T; ++t) {\n            long n"),
    "layout wrong partition width": ("int per = E / P;", "int per = (E / P > 1) ? E / P - 1 : 1;"),
    "capacity drops one too many": ("} else if (rank < cap) {", "} else if (rank + 1 < cap) {"),
    "fp8 ties away from zero": ("code = (c % 2 == 0) ? c : c + 1;", "code = c + 1;"),
    "fp8 scale constant": ("floor_amax / 448.0f", "floor_amax / 447.0f"),
    "fp8 multiply by reciprocal": ("bf16_bits_to_f32(xb[i]) / s;", "bf16_bits_to_f32(xb[i]) * (1.0f / s);"),
    "fp8 no saturation": ("return (uint8_t)(sign | 0x7E);", "return (uint8_t)(sign | 0x7F);"),
    "fp8 wrong block scale": ("recv_s[slot * nb + b] = s;", "recv_s[slot * nb + (b + 1) % nb] = s;"),
    "bf16 rounds ties up": ("(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    "ue8m0 rounds the scale down": ("float s = (mant == 0.5f) ? v : ldexpf(1.0f, ev);",
                                    "float s = (mant == 0.5f) ? v : ldexpf(1.0f, ev - 1);"),
    "ue8m0 exponent bias": ("uint8_t e8 = (uint8_t)(es - 1 + 127);", "uint8_t e8 = (uint8_t)(es + 127);"),
    "fp8 combine wrong scale block": ("s = ((const float *)ys)[slot * nb + i / 128];", "s = ((const float *)ys)[slot * nb];"),
    "combine_src ignores the top-k position": ("if (src_token[r] == t && src_k[r] == j) {",
                                               "if (src_token[r] == t) {"),
    "combine_src ignores the row weight": ("float w = row_w ? row_w[r] : 1.0f;", "float w = 1.0f;"),
    "fp8 combine ue8m0 bias": ("(int)((const uint8_t *)ys)[slot * nb + i / 128] - 127)",
                               "(int)((const uint8_t *)ys)[slot * nb + i / 128] - 126)"),
}

CHECKS = [
    "pl.test_golden_layout_example",
    "lambda: pl.test_random_against_argsort(64, 16, 4, 4, 0.1)",
    "lambda: pl.test_random_against_argsort(333, 256, 8, 32, 0.05)",
    "pf.test_golden_rounding_table",
    "pf.test_golden_fp8_examples",
    "pf.test_midpoints_and_neighbours_match_torch",
    "pf.test_saturation_by_definition",
    "pf.test_golden_ue8m0_examples",
    "pf.test_ue8m0_scale_properties_and_codes_match_torch",
    "pf.test_fp8_dispatch_error_bound_and_amax_code",
    "pc.test_golden_combine_example",
    "pc.test_golden_combine_fp8_example",
    "pc.test_golden_combine_src_example",
    "pc.test_combine_fp8_against_fp64_within_bound",
    "pc.test_combine_against_fp64_within_bound",
    "pc.test_bf16_rounding_matches_torch",
]

_RUNNER = """
import ctypes, json, sys
import oracle
import test_oracle_combine as pc, test_oracle_fp8 as pf, test_oracle_layout as pl
lib_path, checks = sys.argv[1], json.loads(sys.argv[2])
if lib_path:
    real = oracle._load()
    mutant = ctypes.CDLL(lib_path)
    for fn in ("oracle_layout", "oracle_dispatch_bf16", "oracle_dispatch_fp8", "oracle_dispatch_fp8_ue8m0", "oracle_combine", "oracle_combine_fp8",
               "oracle_e4m3_encode_n", "oracle_f32_to_bf16_n", "oracle_e4m3_value"):
        getattr(mutant, fn).restype = getattr(real, fn).restype
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
    oracle._lib = mutant
failed = []
for c in checks:
    try:
        eval(c)()
    except (AssertionError, ValueError, IndexError):
        failed.append(c)
print(json.dumps(failed))
"""


def _run_checks(lib_path: str) -> list:
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([here, os.path.dirname(here)]))
    res = subprocess.run([sys.executable, "-c", _RUNNER, lib_path, json.dumps(CHECKS)],
                         cwd=here, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1])



def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(lib), str(path), "-lm"])
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    caught = _run_checks(_build_mutant(tmp_path, old, new))
    assert caught, f"no pin caught: {name}"


def test_unmutated_oracle_passes_every_check():
    assert _run_checks("") == []
