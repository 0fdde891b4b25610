"""Pins for the oracle's combine and bf16 dispatch.

Pinned against: the hand-worked example in golden/combine_example.txt; an
fp64 recomputation with numpy inside the error bound derived from the
arithmetic (fp32 products and sums, one bf16 rounding); identity experts with
weights whose partial sums are exact (result must equal x bit for bit); and
the bit-copy invariant of bf16 dispatch.  The combine addressed through the
expert-side source maps is pinned by its own hand-worked example (packed,
unweighted and capacity maps), the fp64 bound with the inverse map rebuilt in
numpy, and bit equality with the slot_of combine on oracle layouts.
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


# ---- combine over fp8 expert outputs ----

def _read_fp8_combine_fixture():
    from conftest import read_golden_rows
    rows, slots, weights, out = [], None, None, None
    for r in read_golden_rows("combine_fp8_example.txt"):
        if r[0] == "slots":
            slots = np.array([int(v) for v in r[1:]], np.int32).reshape(2, 2)
        elif r[0] == "weights":
            weights = np.array([float(v) for v in r[1:]], np.float32).reshape(2, 2)
        elif r[0] == "out":
            out = np.array([float(v) for v in r[1:]], np.float64).reshape(2, 2)
        else:
            rows.append((int(r[0]), float(r[1]), int(r[2], 16), int(r[3], 16)))
    yq = np.zeros((3, 128), np.uint8)
    ys = np.zeros((3, 1), np.float32)
    for row, sc, c0, c1 in rows:
        yq[row, 0], yq[row, 1], ys[row, 0] = c0, c1, sc
    return yq, ys, slots, weights, out


def test_golden_combine_fp8_example():
    yq, ys, slots, w, expect = _read_fp8_combine_fixture()
    got = oracle.bf16_to_f32(oracle.combine_fp8(yq, ys, w, slots))[:, :2]
    np.testing.assert_array_equal(got.astype(np.float64), expect)
    # the same scales as UE8M0 exponents give the same result (they are powers of two)
    e8 = (np.log2(ys).astype(np.int64) + 127).astype(np.uint8)
    got8 = oracle.bf16_to_f32(oracle.combine_fp8(yq, e8, w, slots))[:, :2]
    np.testing.assert_array_equal(got8.astype(np.float64), expect)


def test_combine_fp8_against_fp64_within_bound():
    import torch
    rng = np.random.default_rng(23)
    T, H, k, R = 40, 384, 6, 300
    yq = rng.integers(0, 256, size=(R, H)).astype(np.uint8)
    yq[(yq & 0x7F) == 0x7F] = 0x11                               # no NaN codes
    ys = np.exp(rng.uniform(-6, 6, size=(R, H // 128))).astype(np.float32)
    w = rng.standard_normal((T, k)).astype(np.float32)
    slot_of = rng.integers(0, R, size=(T, k)).astype(np.int32)
    slot_of[rng.random((T, k)) < 0.2] = -1
    out = oracle.combine_fp8(yq, ys, w, slot_of)
    table = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vals = table[yq] * np.repeat(ys.astype(np.float64), 128, axis=1)      # [R, H]
    valid = slot_of >= 0
    rows = vals[np.where(valid, slot_of, 0)]
    wv = np.where(valid, w.astype(np.float64), 0.0)[:, :, None]
    exact = (wv * rows).sum(axis=1)
    mag = (np.abs(wv) * np.abs(rows)).sum(axis=1)
    err32 = 3 * k * 2.0 ** -24 * mag                               # dequant, product and sum roundings
    bound = 2.0 ** -8 * (np.abs(exact) + err32) + err32
    got = oracle.bf16_to_f32(out).astype(np.float64)
    assert (np.abs(got - exact) <= bound * (1 + 1e-9) + 1e-300).all()
    # unweighted = weights of one
    np.testing.assert_array_equal(oracle.combine_fp8(yq, ys, None, slot_of),
                                  oracle.combine_fp8(yq, ys, np.ones_like(w), slot_of))


def test_fp8_dispatch_then_fp8_combine_returns_x_within_quantisation():
    d = W.make(W.WORKLOADS["decode"].shrink(16))
    wl = d["wl"]
    L = oracle.layout(d["topk_idx"], wl.E, wl.P, oracle.CAPACITY, wl.capacity)
    q, s, _ = oracle.dispatch_fp8(d["x"], L["slot_of"], wl.R)
    w = np.full((wl.T, wl.k), 1.0 / wl.k, np.float32)             # exact: k = 8
    out = oracle.bf16_to_f32(oracle.combine_fp8(q, s, w, L["slot_of"])).astype(np.float64)
    x = oracle.bf16_to_f32(d["x"]).astype(np.float64)
    sb = np.repeat(s[L["slot_of"][:, 0]].astype(np.float64), 128, axis=1)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * sb) * 1.0001 + 2.0 ** -8 * np.abs(x) + 1e-30
    assert (np.abs(out - x) <= bound).all()


# ---- combine addressed from the expert side (src_token / src_k, per-row weights)

def test_golden_combine_src_example():
    g = read_golden_kv("combine_src_example.txt")
    H, T, k = (int(g[n][0]) for n in ("H", "T", "k"))
    y = W.to_bf16_bits(floats(g["y"]).reshape(-1, H).astype(np.float32))
    for prefix, wkey, outkey in (("", "row_w", "out"), ("", None, "out_unweighted"), ("cap_", "cap_row_w", "cap_out")):
        st = ints(g[prefix + "src_token"]).astype(np.int32)
        sk = ints(g[prefix + "src_k"]).astype(np.int32)
        rw = None if wkey is None else floats(g[wkey]).astype(np.float32)
        out = oracle.combine_src(y, rw, st, sk, T, k)
        np.testing.assert_array_equal(oracle.bf16_to_f32(out).ravel(), floats(g[outkey]).astype(np.float32),
                                      err_msg=outkey)


def _inverse_maps(src_token, src_k, T, k):
    """slot[t, j] = the row holding (t, j), -1 if none (numpy, independent of the C code)."""
    slot = np.full((T, k), -1, np.int32)
    live = np.nonzero(src_token >= 0)[0]
    slot[src_token[live], src_k[live]] = live
    return slot


def test_combine_src_against_fp64_within_bound():
    rng = np.random.default_rng(21)
    for T, H, k, R, drop in [(40, 48, 8, 500, 0.2), (9, 8, 1, 12, 0.0), (25, 16, 5, 200, 0.5)]:
        # a random injective placement of the live (t, j) pairs into R rows
        pairs = [(t, j) for t in range(T) for j in range(k) if rng.random() >= drop]
        rows = rng.permutation(R)[: len(pairs)]
        src_token = np.full(R, -1, np.int32)
        src_k = np.full(R, -1, np.int32)
        for (t, j), r in zip(pairs, rows):
            src_token[r], src_k[r] = t, j
        y = W.to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32) * 2)
        row_w = rng.standard_normal(R).astype(np.float32)
        out = oracle.combine_src(y, row_w, src_token, src_k, T, k)
        slot = _inverse_maps(src_token, src_k, T, k)
        w = np.where(slot >= 0, row_w[np.maximum(slot, 0)], 0).astype(np.float32)
        _fp64_bound_check(y, w, slot, out)


def test_combine_src_equals_slot_combine_on_layouts():
    """Rows found through the expert-side maps give exactly the slot_of combine
    (same products, same j order), packed and capacity, with masked copies."""
    rng = np.random.default_rng(8)
    for T, E, k, P, cap, mask in [(100, 16, 4, 4, None, 0.1), (64, 8, 8, 2, 40, 0.0), (30, 32, 3, 8, 2, 0.2)]:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
        idx[rng.random((T, k)) < mask] = -1
        if cap is None:
            L = oracle.layout(idx, E, P)
            R = T * k
        else:
            L = oracle.layout(idx, E, P, mode=oracle.CAPACITY, cap=cap)
            R = E * cap
        H = 24
        y = W.to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
        topk_w = rng.random((T, k)).astype(np.float32)
        st, sk = L["src_token"], L["src_k"]
        row_w = np.where(st >= 0, topk_w[np.maximum(st, 0), np.maximum(sk, 0)], 7.0).astype(np.float32)
        np.testing.assert_array_equal(oracle.combine_src(y, row_w, st, sk, T, k),
                                      oracle.combine(y, topk_w, L["slot_of"]))
        np.testing.assert_array_equal(oracle.combine_src(y, None, st, sk, T, k),
                                      oracle.combine(y, np.ones((T, k), np.float32), L["slot_of"]))
        # the row order of the expert-side buffer does not matter
        p = rng.permutation(R)
        np.testing.assert_array_equal(oracle.combine_src(y[p], row_w[p], st[p], sk[p], T, k),
                                      oracle.combine(y, topk_w, L["slot_of"]))
