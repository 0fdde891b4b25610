"""GPU combine addressed by the expert-side source maps (ep_combine_src) vs the
CPU oracle, through the C ABI.

The maps and every other input come from the oracle's own layout and the
seeded generators; the bar is the combine tolerance
|gpu - oracle| <= 1e-2 + 1e-2 * |oracle| (bf16), and bit equality (same
operation order as the oracle).  Also checked: the output is
bit-identical to ep_combine / ep_combine_fp8 given the equivalent slot_of and
weights, whatever the workspace held before the call (garbage, or the map of
an earlier call with other routing), and bad pairs are skipped and flagged.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_04_gb300 as ep
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

RTOL = ATOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    ep.load()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(b: np.ndarray) -> torch.Tensor:
    return dev(b.view(np.int16)).view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_combine_close(g_bits: np.ndarray, o_bits: np.ndarray):
    """The tolerance contract, then bit equality."""
    g = oracle.bf16_to_f32(g_bits).astype(np.float64)
    o = oracle.bf16_to_f32(o_bits).astype(np.float64)
    diff = np.abs(g - o)
    bad = diff > ATOL + RTOL * np.abs(o)
    assert not bad.any(), f"{bad.sum()} elements out of tolerance, max |diff| {diff.max()}"
    n_diff = int((g_bits != o_bits).sum())
    assert n_diff == 0, f"{n_diff} elements differ in their bits (max |diff| {diff.max()}, within tolerance)"


def _routing(rng, T, E, k, mask):
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < mask] = -1
    return idx


def _case(T, H, E, k, cap, mask, seed):
    rng = np.random.default_rng(seed)
    idx = _routing(rng, T, E, k, mask)
    if cap is None:
        L = oracle.layout(idx, E, 1)
    else:
        L = oracle.layout(idx, E, 1, oracle.CAPACITY, cap)
    R = L["src_token"].shape[0]
    y = W.to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32) * 2)
    topk_w = rng.random((T, k)).astype(np.float32)
    st, sk = L["src_token"], L["src_k"]
    # each row carries the weight of the copy it holds; rows without a copy get a
    # value that must not matter
    row_w = np.where(st >= 0, topk_w[np.maximum(st, 0), np.maximum(sk, 0)], 5.0).astype(np.float32)
    return rng, idx, L, y, topk_w, row_w


def _plan(T, H, E, k, cap):
    return ep.Plan(T, H, E, k, 1, cap)


SHAPES = [
    (128, 1024, 16, 4, None, 0.0),       # tiny-shaped, packed
    (128, 7168, 256, 8, 128, 0.0),       # decode-shaped capacity buffer, 1024 of 32768 rows live
    (1, 8, 2, 1, None, 0.0),
    (37, 264, 8, 8, None, 0.2),          # k = E, masked copies, a ragged 528-byte row
    (300, 1024, 32, 6, 20, 0.1),         # capacity overflow: dropped copies
    (2000, 512, 64, 8, None, 0.0),       # more units than resident CTAs (persistent ring)
    (20, 512, 64, 32, None, 0.1),        # top-32: 32 rows a unit, masked copies
]


@pytest.mark.parametrize("T,H,E,k,cap,mask", SHAPES)
@pytest.mark.parametrize("weighted", [True, False])
def test_combine_src_matches_oracle(T, H, E, k, cap, mask, weighted):
    rng, idx, L, y, topk_w, row_w = _case(T, H, E, k, cap, mask, T * 7 + H + k)
    plan = _plan(T, H, E, k, cap)
    rw = row_w if weighted else None
    out = plan.combine_src(bf16_dev(y), None if rw is None else dev(rw), dev(L["src_token"]), dev(L["src_k"]))
    got = bits(out)
    assert_combine_close(got, oracle.combine_src(y, rw, L["src_token"], L["src_k"], T, k))
    # bit-identical to the slot_of combine with the same weights
    ref = plan.combine(bf16_dev(y), dev(topk_w) if weighted else None, out=torch.empty_like(out),
                       slot_of=dev(L["slot_of"]))
    np.testing.assert_array_equal(got, bits(ref))
    assert int(plan.layout_out.err_flags.item()) == 0


# Whatever the workspace held must not matter, for the one-unit gather (the
# first two shapes) and the ring (the last): in-range row numbers of rows that
# hold other pairs, out-of-range values, maps of earlier calls with other
# routing, with masked and dropped copies leaving pairs that no row claims.
@pytest.mark.parametrize("T,H,E,k,cap", [(300, 256, 32, 6, 20), (128, 7168, 256, 8, 128), (2000, 512, 64, 8, 300)])
def test_combine_src_ignores_what_the_workspace_held(T, H, E, k, cap):
    plan = _plan(T, H, E, k, cap)
    g = torch.Generator(device="cuda").manual_seed(3)
    plan.src_workspace.view(torch.int32)[:] = torch.randint(-2, plan.R + 2, (plan.src_workspace.numel() // 4,),
                                                           generator=g, device="cuda", dtype=torch.int32)
    for seed in (11, 12, 13):              # each call leaves a map the next call must not trust
        _, _, L, y, _, row_w = _case(T, H, E, k, cap, 0.15, seed)
        out = plan.combine_src(bf16_dev(y), dev(row_w), dev(L["src_token"]), dev(L["src_k"]))
        assert_combine_close(bits(out), oracle.combine_src(y, row_w, L["src_token"], L["src_k"], T, k))


@pytest.mark.parametrize("ue8m0", [False, True])
@pytest.mark.parametrize("T,H,E,k,cap", [(128, 7168, 256, 8, 128), (50, 384, 8, 3, None), (700, 1024, 16, 8, None)])
def test_combine_src_fp8_matches_oracle(T, H, E, k, cap, ue8m0):
    rng, idx, L, _, topk_w, row_w = _case(T, H, E, k, cap, 0.05, T + H + ue8m0)
    R = L["src_token"].shape[0]
    q = rng.integers(0, 256, size=(R, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A                                   # no NaN codes
    if ue8m0:
        s = rng.integers(100, 140, size=(R, H // 128)).astype(np.uint8)
    else:
        s = np.exp(rng.uniform(-8, 8, size=(R, H // 128))).astype(np.float32)
    plan = _plan(T, H, E, k, cap)
    g = torch.Generator(device="cuda").manual_seed(T)
    plan.src_workspace.view(torch.int32)[:] = torch.randint(0, R, (plan.src_workspace.numel() // 4,), generator=g,
                                                           device="cuda", dtype=torch.int32)   # stale rows
    out = plan.combine_src(dev(q).view(torch.float8_e4m3fn), dev(row_w), dev(L["src_token"]), dev(L["src_k"]),
                           y_scales=dev(s))
    got = bits(out)
    # the weight each row carries is exactly topk_w of its copy, so the
    # oracle's slot_of combine over fp8 outputs is the expected value
    assert_combine_close(got, oracle.combine_fp8(q, s, topk_w, L["slot_of"]))
    ref = plan.combine_fp8(dev(q).view(torch.float8_e4m3fn), dev(s), dev(topk_w), out=torch.empty_like(out),
                           slot_of=dev(L["slot_of"]))
    np.testing.assert_array_equal(got, bits(ref))


def test_combine_src_bad_pairs_are_skipped_and_flagged():
    T, H, E, k = 64, 128, 16, 4
    _, _, L, y, _, row_w = _case(T, H, E, k, None, 0.0, 77)
    st, sk = L["src_token"].copy(), L["src_k"].copy()
    st[3], sk[10], st[20] = T, k, -5                                # three rows outside [0,T) x [0,k)
    plan = _plan(T, H, E, k, None)
    plan.layout_out.err_flags.zero_()
    out = plan.combine_src(bf16_dev(y), dev(row_w), dev(st), dev(sk))
    assert_combine_close(bits(out), oracle.combine_src(y, row_w, st, sk, T, k))
    assert int(plan.layout_out.err_flags.item()) & ep.ERRF_BAD_SLOT


def test_combine_src_after_gpu_dispatch_round_trip():
    """The whole expert-side path: GPU layout + dispatch (recv_w routed with
    the rows), identity experts, combine through the GPU's own source maps and
    row weights; weights with exact sums return x bit for bit."""
    d = W.make("tiny")
    wl = d["wl"]
    plan = ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, None, with_weights=True)
    w = np.full((wl.T, wl.k), 1.0 / wl.k, np.float32)
    plan.layout(dev(d["topk_idx"]))
    recv, _, recv_w = plan.dispatch(bf16_dev(d["x"]), dev(w))
    out = plan.combine_src(recv, recv_w)
    np.testing.assert_array_equal(bits(out), d["x"])


def _random_bf16_rows(rng, R, H):
    """Finite bf16 bit patterns, magnitudes in [2^-6, 2^2), random signs: cheap at
    full size (one draw of 16-bit integers)."""
    raw = rng.integers(0, 1 << 16, size=(R, H), dtype=np.uint16)
    exp = ((raw >> np.uint16(7)) & np.uint16(0x7)) + np.uint16(121)
    return (raw & np.uint16(0x807F)) | (exp << np.uint16(7))


@pytest.mark.parametrize("name", ["prefill", "skewed", "grouped"])
def test_combine_src_full_size(name):
    """Full-size workload in the benchmark's launch configuration: the oracle's
    layout gives the source maps, seeded numpy the expert outputs and row
    weights.  Every output token equals the slot_of combine bit for bit and the
    oracle's combine by source maps over the whole buffer."""
    d = W.make(name)
    wl = d["wl"]
    L = oracle.layout(d["topk_idx"], wl.E, wl.P)
    rng = np.random.default_rng(17)
    y = _random_bf16_rows(rng, wl.R, wl.H)
    row_w = rng.random(wl.R).astype(np.float32)
    st, sk = L["src_token"], L["src_k"]
    plan = ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, None)
    y_d = bf16_dev(y)
    out = plan.combine_src(y_d, dev(row_w), dev(st), dev(sk)).clone()
    topk_w = np.where(L["slot_of"] >= 0, row_w[np.maximum(L["slot_of"], 0)], 0).astype(np.float32)
    ref = plan.combine(y_d, dev(topk_w), out=torch.empty_like(out), slot_of=dev(L["slot_of"]))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert int(plan.layout_out.err_flags.item()) == 0
    o = oracle.combine_src(y, row_w, st, sk, wl.T, wl.k)
    assert_combine_close(bits(out), o)
