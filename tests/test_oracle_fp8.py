"""Pins for the oracle's FP8 e4m3 encoder and its fp8 dispatch.

Pinned against: torch's float8_e4m3fn conversions (an independent library
implementation of the same format) for every code and for rounding below 464,
exhaustively over every non-negative float32 there (torch does not saturate,
so values >= 464 are pinned by the format definition instead); hand-worked values in golden/; the quantisation error bound of the
format; and the amax code property of every block.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import read_golden_rows


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_code_values_match_torch():
    table = oracle.e4m3_table()
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(table) == nan).all() and nan.sum() == 2
    np.testing.assert_array_equal(table[~nan], ref[~nan])
    assert np.nanmax(table) == 448.0 and table[1] == 2.0 ** -9


def test_golden_rounding_table():
    for value, code in read_golden_rows("e4m3_rounding.txt"):
        got = oracle.e4m3_encode(np.array([float(value)], np.float32))[0]
        assert got == int(code, 16), (value, hex(got), code)


def test_golden_fp8_examples():
    for amax, s_bits, x, code in read_golden_rows("fp8_examples.txt"):
        # a 128-block holding x and amax (all other channels 0)
        xs = np.zeros((1, 128), np.float32)
        xs[0, 0] = float(amax)
        xs[0, 1] = float(x)
        xb = W.to_bf16_bits(xs)
        assert oracle.bf16_to_f32(xb)[0, 1] == np.float32(float(x))
        q, s, _ = oracle.dispatch_fp8(xb, np.array([[0]], np.int32), 1)
        assert s[0, 0].view(np.uint32) == int(s_bits, 16), (amax, hex(s[0, 0].view(np.uint32)))
        assert q[0, 1] == int(code, 16), (amax, x, hex(q[0, 1]))


def test_midpoints_and_neighbours_match_torch():
    """Every rounding boundary of the format, and one float either side."""
    table = oracle.e4m3_table()[:0x7F]             # non-negative finite codes
    mids = ((table[:-1] + table[1:]) / 2).astype(np.float32)
    pts = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                          np.nextafter(mids, np.float32(0)), table.astype(np.float32)])
    pts = pts[pts < 464.0]
    pts = np.concatenate([pts, -pts])
    np.testing.assert_array_equal(oracle.e4m3_encode(pts), _torch_e4m3(pts))


def test_random_and_one_binade_exhaustive_match_torch():
    rng = np.random.default_rng(7)
    v = (2.0 ** rng.uniform(-16, np.log2(464.0), size=2_000_000)).astype(np.float32)
    v = v[v < 464.0]
    v *= np.where(rng.random(v.shape) < 0.5, -1, 1).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), _torch_e4m3(v))
    # every float32 in [1, 2) and in the subnormal-rounding range [2^-10, 2^-9)
    for lo in (1.0, 2.0 ** -10):
        base = np.float32(lo).view(np.uint32)
        bits = np.arange(base, base + (1 << 23), dtype=np.uint32)
        vals = bits.view(np.float32)
        np.testing.assert_array_equal(oracle.e4m3_encode(vals), _torch_e4m3(vals))


def _sweep_e4m3(bounds):
    """Oracle vs torch codes for every float32 bit pattern in [lo, hi), and for
    the negatives of every 17th of them; (mismatches, first mismatching bits)."""
    lo, hi = bounds
    bits = np.arange(lo, hi, dtype=np.uint32)
    v = bits.view(np.float32)
    bad = np.flatnonzero(oracle.e4m3_encode(v) != _torch_e4m3(v))
    neg = -v[::17]
    bad_neg = np.flatnonzero(oracle.e4m3_encode(neg) != _torch_e4m3(neg))
    first = int(bits[bad[0]]) if bad.size else (int(bits[::17][bad_neg[0]]) | 0x80000000 if bad_neg.size else -1)
    return int(bad.size + bad_neg.size), first


def test_every_float32_below_464_matches_torch():
    """Exhaustive: each of the 1.14e9 non-negative float32 values below 464
    (where torch's conversion rounds without saturating) gets torch's code,
    i.e. the nearest code with ties to even; negatives on a stride."""
    import multiprocessing as mp
    end = int(np.float32(464.0).view(np.uint32))
    step = 1 << 26
    ranges = [(lo, min(end, lo + step)) for lo in range(0, end, step)]
    with mp.get_context("spawn").Pool(min(len(ranges), max(1, len(os.sched_getaffinity(0))))) as pool:
        results = pool.map(_sweep_e4m3, ranges, chunksize=1)
    n_bad = sum(r[0] for r in results)
    firsts = [r[1] for r in results if r[0]]
    assert n_bad == 0, f"{n_bad} float32 values encode differently, first at bits {firsts[0]:#010x}"


def test_saturation_by_definition():
    big = np.array([448.0, 448.5, 463.9, 464.0, 464.1, 1e6, 3.4e38, np.inf], np.float32)
    assert (oracle.e4m3_encode(big) == 0x7E).all()
    assert (oracle.e4m3_encode(-big) == 0xFE).all()


def _dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    table = oracle.e4m3_table()
    H = q.shape[1]
    return table[q] * np.repeat(s.astype(np.float64), 128, axis=1)[:, :H]


def test_fp8_dispatch_error_bound_and_amax_code():
    rng = np.random.default_rng(3)
    T, H, k, E = 37, 512, 3, 5
    xf = rng.standard_normal((T, H)).astype(np.float32) * np.exp(rng.uniform(-6, 6, (T, 1))).astype(np.float32)
    x = W.to_bf16_bits(xf)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    L = oracle.layout(idx, E, 1)
    R = T * k
    q, s, _ = oracle.dispatch_fp8(x, L["slot_of"], R)
    xr = oracle.bf16_to_f32(x).astype(np.float64)
    for t in range(T):
        rows = L["slot_of"][t]
        for r in rows:                                   # k identical copies
            np.testing.assert_array_equal(q[r], q[rows[0]])
            np.testing.assert_array_equal(s[r], s[rows[0]])
        deq = _dequant(q[rows[0]][None], s[rows[0]][None])[0]
        sb = np.repeat(s[rows[0]].astype(np.float64), 128)
        # half an e4m3 ulp: 2^-4 relative for normals, 2^-10 * s absolute for subnormals
        bound = np.maximum(2.0 ** -4 * np.abs(xr[t]), 2.0 ** -10 * sb) * (1 + 1e-5)
        assert (np.abs(deq - xr[t]) <= bound).all()
        # the amax element of each block maps to +-448 (code 0x7E / 0xFE)
        for b in range(H // 128):
            blk = xr[t, b * 128:(b + 1) * 128]
            i = np.argmax(np.abs(blk))
            assert q[rows[0], b * 128 + i] & 0x7F == 0x7E
            assert np.float32(s[rows[0], b]) == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))


def test_fp8_all_zero_block_and_untouched_rows():
    x = np.zeros((2, 256), np.uint16)
    x[1, 128:] = W.to_bf16_bits(np.linspace(-3, 3, 128, dtype=np.float32))
    slot_of = np.array([[2], [0]], np.int32)
    q, s, _ = oracle.dispatch_fp8(x, slot_of, 4)
    assert (q[2] == 0).all()
    assert s[2, 0] == np.float32(1e-4) / np.float32(448.0) and s[2, 1] == s[2, 0]
    assert (q[0, :128] == 0).all() and q[0, 128:].max() > 0
    assert (q[1] == 0).all() and (s[1] == 0).all() and (q[3] == 0).all()    # no copy there


def test_fp8_rejects_bad_hidden():
    with pytest.raises(ValueError):
        oracle.dispatch_fp8(np.zeros((1, 100), np.uint16), np.zeros((1, 1), np.int32), 1)


# ---- exact-rational restatement of the quantisation, independent of the C code ----

def _rn32(fr: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (exact)."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


_E4M3 = [Fraction(c & 7, 512) if (c >> 3) == 0 else (1 + Fraction(c & 7, 8)) * Fraction(2) ** ((c >> 3) - 7)
         for c in range(0x7F)]


def _e4m3_exact(fr: Fraction) -> int:
    sign = 0x80 if fr < 0 else 0
    a = abs(fr)
    if a >= 448:
        return sign | 0x7E
    c = max(i for i, v in enumerate(_E4M3) if v <= a)
    twice, mid = 2 * a, _E4M3[c] + _E4M3[c + 1]
    code = c if twice < mid else c + 1 if twice > mid else (c if c % 2 == 0 else c + 1)
    return sign | code


def _distinguishing_inputs(n_amax: int):
    """Inputs where x/s and x*(1/s) round to different e4m3 codes (found by search)."""
    rng = np.random.default_rng(0)
    amax = oracle.bf16_to_f32(W.to_bf16_bits(np.abs(rng.standard_normal(n_amax)).astype(np.float32) * 3 + 0.1))
    xs = oracle.bf16_to_f32(W.to_bf16_bits(rng.standard_normal(20000).astype(np.float32)))
    pairs = []
    for a in amax:
        s = np.float32(a) / np.float32(448)
        cand = xs[np.abs(xs) <= a]
        d = oracle.e4m3_encode(cand / s) != oracle.e4m3_encode(cand * (np.float32(1) / s))
        pairs += [(float(a), float(v)) for v in cand[d][:2]]
    return pairs


def test_fp8_matches_exact_rational_definition():
    """s = RN32(amax/448), q = e4m3(RN32(x/s)) recomputed with exact rationals."""
    rng = np.random.default_rng(21)
    pairs = _distinguishing_inputs(300)
    assert len(pairs) >= 10
    # pack each (amax, x) into its own 128-block, plus some random full blocks
    blocks = []
    for a, v in pairs:
        blk = np.zeros(128, np.float32)
        blk[0], blk[1] = a, v
        blocks.append(blk)
    for _ in range(8):
        blocks.append((rng.standard_normal(128) * np.exp(rng.uniform(-8, 8))).astype(np.float32))
    x = W.to_bf16_bits(np.stack(blocks).reshape(-1, 256))
    T = x.shape[0]
    q, s, _ = oracle.dispatch_fp8(x, np.arange(T, dtype=np.int32)[:, None], T)
    xf = oracle.bf16_to_f32(x)
    for t in range(T):
        for b in range(2):
            blk = xf[t, b * 128:(b + 1) * 128]
            amax = max(Fraction(float(abs(v))) for v in blk)
            s_exact = _rn32(max(amax, Fraction(float(np.float32(1e-4)))) / 448)
            assert Fraction(float(s[t, b])) == s_exact
            for i in range(128):
                assert q[t, b * 128 + i] == _e4m3_exact(_rn32(Fraction(float(blk[i])) / s_exact)), (t, b, i)


# ---- UE8M0 (power-of-two) scales ----

def test_golden_ue8m0_examples():
    for amax, e8, x, code in read_golden_rows("ue8m0_examples.txt"):
        xs = np.zeros((1, 128), np.float32)
        xs[0, 0] = float(amax)
        xs[0, 1] = float(x)
        q, e, _ = oracle.dispatch_fp8_ue8m0(W.to_bf16_bits(xs), np.array([[0]], np.int32), 1)
        assert e[0, 0] == int(e8), (amax, e[0, 0])
        assert q[0, 1] == int(code, 16), (amax, x, hex(q[0, 1]))


def test_ue8m0_scale_properties_and_codes_match_torch():
    """s is a power of two with v <= s < 2v; codes equal torch's e4m3 of x/s."""
    rng = np.random.default_rng(17)
    T, H = 64, 1024
    xf = (rng.standard_normal((T, H // 128, 128)) * np.exp(rng.uniform(-14, 10, (T, H // 128, 1)))).reshape(T, H)
    xf = xf.astype(np.float32)
    xf[3, :128] = 0.0
    x = W.to_bf16_bits(xf)
    q, e, _ = oracle.dispatch_fp8_ue8m0(x, np.arange(T, dtype=np.int32)[:, None], T)
    q32, s32, _ = oracle.dispatch_fp8(x, np.arange(T, dtype=np.int32)[:, None], T)
    s = oracle.ue8m0_value(e)                                     # float64, exact powers of two
    v = s32.astype(np.float64)                                    # RN32(max(amax,1e-4)/448)
    assert (s >= v).all() and (s < 2 * v).all()
    assert (np.frexp(s)[0] == 0.5).all()
    xr = oracle.bf16_to_f32(x).astype(np.float64)
    quot = (xr / np.repeat(s, 128, axis=1)).astype(np.float32)     # exact: s is a power of two
    assert (np.abs(quot) <= 448.0).all()
    np.testing.assert_array_equal(q, _torch_e4m3(quot))
    assert (q[3, :128] == 0).all() and e[3, 0] == 105
