"""Pins for the oracle's combine and bf16 dispatch.

Pinned against: the hand-worked example in golden/combine_example.txt; an
fp64 recomputation with numpy inside the error bound derived from the
arithmetic (fp32 products and sums, one bf16 rounding); identity experts with
weights whose partial sums are exact (result must equal x bit for bit); and
the bit-copy invariant of bf16 dispatch.
"""
import numpy as np
import torch

import oracle
import workloads as W
from conftest import floats, ints, read_golden_kv


def test_golden_combine_example():
    g = read_golden_kv("combine_example.txt")
    H = int(g["H"][0])
    slot_of = ints(g["slot_of"]).reshape(-1, 2).astype(np.int32)
    w = floats(g["topk_w"]).reshape(-1, 2).astype(np.float32)
    y = W.to_bf16_bits(floats(g["y"]).reshape(-1, H).astype(np.float32))
    out = oracle.combine(y, w, slot_of)
    np.testing.assert_array_equal(oracle.bf16_to_f32(out).ravel(), floats(g["out"]).astype(np.float32))


def _fp64_bound_check(y, w, slot_of, out):
    yf = oracle.bf16_to_f32(y).astype(np.float64)
    T, k = slot_of.shape
    valid = slot_of >= 0
    rows = yf[np.where(valid, slot_of, 0)]                       # [T, k, H]
    wv = np.where(valid, w.astype(np.float64), 0.0)[:, :, None]
    exact = (wv * rows).sum(axis=1)
    mag = (np.abs(wv) * np.abs(rows)).sum(axis=1)
    err32 = 2 * k * 2.0 ** -24 * mag                            # fp32 products + k sums
    bound = 2.0 ** -8 * (np.abs(exact) + err32) + err32          # + one bf16 rounding
    got = oracle.bf16_to_f32(out).astype(np.float64)
    assert (np.abs(got - exact) <= bound * (1 + 1e-9) + 1e-300).all()
    return np.abs(got - exact).max()


def test_combine_against_fp64_within_bound():
    rng = np.random.default_rng(11)
    for T, H, k, R, mask in [(50, 64, 8, 400, 0.1), (7, 8, 1, 7, 0.0), (20, 24, 5, 300, 0.3)]:
        y = W.to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32) * 3)
        w = rng.standard_normal((T, k)).astype(np.float32)
        slot_of = rng.integers(0, R, size=(T, k)).astype(np.int32)
        slot_of[rng.random((T, k)) < mask] = -1
        out = oracle.combine(y, w, slot_of)
        _fp64_bound_check(y, w, slot_of, out)
        # a token whose slots are all masked gives exactly 0
        slot_of[0, :] = -1
        assert (oracle.combine(y, w, slot_of)[0] == 0).all()


def test_combine_order_matters_only_through_rounding():
    """Permuting j changes at most the last bf16 bit (same exact sum)."""
    rng = np.random.default_rng(5)
    T, H, k, R = 40, 32, 8, 320
    y = W.to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    w = rng.random((T, k)).astype(np.float32)
    slot_of = rng.permutation(R)[: T * k].reshape(T, k).astype(np.int32)
    a = oracle.bf16_to_f32(oracle.combine(y, w, slot_of))
    p = rng.permutation(k)
    b = oracle.bf16_to_f32(oracle.combine(y, w[:, p], slot_of[:, p]))
    np.testing.assert_allclose(a, b, rtol=2 ** -7, atol=1e-6)


def test_identity_experts_round_trip():
    d = W.make(W.WORKLOADS["tiny"])
    wl = d["wl"]
    L = oracle.layout(d["topk_idx"], wl.E, wl.P)
    recv, recv_w = oracle.dispatch_bf16(d["x"], L["slot_of"], wl.R, d["topk_w"])
    # bf16 dispatch is a bit copy into every routed row, and routes the weights
    for t in range(wl.T):
        for j in range(wl.k):
            s = L["slot_of"][t, j]
            np.testing.assert_array_equal(recv[s], d["x"][t])
            assert recv_w[s] == d["topk_w"][t, j]
    # weights with exact partial sums (powers of two, total 1): out == x exactly
    w_exact = np.tile(np.array([0.5, 0.25, 0.125, 0.125], np.float32), (wl.T, 1))
    np.testing.assert_array_equal(oracle.combine(recv, w_exact, L["slot_of"]), d["x"])
    # softmax weights (sum 1 within a few fp32 ulps): within the combine tolerance
    out = oracle.bf16_to_f32(oracle.combine(recv, d["topk_w"], L["slot_of"]))
    x = oracle.bf16_to_f32(d["x"])
    assert (np.abs(out - x) <= 1e-2 + 1e-2 * np.abs(x)).all()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(1_000_000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 1_000_000).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-45, -1e-45, 1.17549435e-38], np.float32),
        # exact ties: bf16 value + half a bf16 ulp, both parities
        (np.arange(0x3F800000, 0x3F800000 + 4096, dtype=np.uint32) * 0 + 0x3F800000 + np.arange(4096, dtype=np.uint32) * 0x10000 + 0x8000).view(np.float32),
    ])
    v = v[np.isfinite(v) | np.isinf(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16(v), ref)
    assert oracle.f32_to_bf16(np.array([np.nan], np.float32))[0] & 0x7FC0 == 0x7FC0


def test_dispatch_bf16_leaves_other_rows_untouched():
    x = np.arange(12, dtype=np.uint16).reshape(3, 4)
    slot_of = np.array([[4, -1], [0, 2], [-1, -1]], np.int32)
    sentinel = np.full((6, 4), 0xBEEF, np.uint16)
    recv, _ = oracle.dispatch_bf16(x, slot_of, 6, recv=sentinel)
    np.testing.assert_array_equal(recv[4], x[0])
    np.testing.assert_array_equal(recv[0], x[1])
    np.testing.assert_array_equal(recv[2], x[1])
    for r in (1, 3, 5):
        assert (recv[r] == 0xBEEF).all()
