"""GPU path vs the CPU oracle, through the C ABI (via the ctypes binding).

Bar: layout, indices, bf16 receive rows and the fp8 payload + scales are
bit-exact; combine is within |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| (bf16),
the documented contract, and is also asserted bit-equal: the kernel adds the
same fp32 products in the same j order with the same roundings as the oracle,
so any difference would mean a reordered or contracted operation.
Sizes: every workload at full size with whole outputs compared (the largest,
group-limited, moves 2.4 GB per step), shrunken workloads, random shapes
crossing every tile and chunk boundary, and the degenerate cases (T = 0,
T = 1, k = 1, k = E, all copies to one expert, capacity overflow, bad ids,
all-zero blocks).
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


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return dev(bits.view(np.int16)).view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def plan_for(wl: W.Workload, with_weights=False) -> ep.Plan:
    cap = wl.capacity if wl.mode == W.CAPACITY else None
    return ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, cap, fp8=wl.fp8, with_weights=with_weights)


def oracle_layout(wl: W.Workload, idx: np.ndarray) -> dict:
    mode = oracle.CAPACITY if wl.mode == W.CAPACITY else oracle.PACKED
    return oracle.layout(idx, wl.E, wl.P, mode, wl.capacity)


def gpu_layout(plan: ep.Plan, idx: np.ndarray) -> dict:
    L = plan.layout(dev(idx))
    torch.cuda.synchronize()
    out = {k: getattr(L, k).cpu().numpy() for k in
           ("counts", "offsets", "part_counts", "part_offsets", "slot_of", "src_token", "src_k")}
    out["err"] = int(L.err_flags.cpu().numpy().view(np.uint32)[0])
    return out


def assert_layout_equal(g: dict, o: dict):
    for key in ("counts", "offsets", "part_counts", "part_offsets", "slot_of", "src_token", "src_k"):
        np.testing.assert_array_equal(g[key], o[key], err_msg=key)
    assert g["err"] == o["err"]


def assert_combine_close(g_bits: np.ndarray, o_bits: np.ndarray):
    """The tolerance contract, then bit equality (the kernel keeps the oracle's
    operation order, so a difference is a finding, not rounding noise)."""
    g = oracle.bf16_to_f32(g_bits).astype(np.float64)
    o = oracle.bf16_to_f32(o_bits).astype(np.float64)
    diff = np.abs(g - o)
    bad = diff > ATOL + RTOL * np.abs(o)
    assert not bad.any(), f"{bad.sum()} elements out of tolerance, max |diff| {diff.max()}"
    n_diff = int((g_bits != o_bits).sum())
    assert n_diff == 0, f"{n_diff} elements differ in their bits (max |diff| {diff.max()}, within tolerance)"


# ------------------------------------------------------------------ layout

@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_layout_workloads_full_size(name):
    d = W.make(name)
    wl = d["wl"]
    assert_layout_equal(gpu_layout(plan_for(wl), d["topk_idx"]), oracle_layout(wl, d["topk_idx"]))


LAYOUT_FUZZ = [
    # (T, E, k, P, capacity or None, mask_frac, duplicates allowed)
    (1, 1, 1, 1, None, 0.0, False), (1, 16, 16, 4, None, 0.0, False), (3, 5, 2, 1, 1, 0.2, True),
    (31, 7, 1, 7, None, 0.0, False), (33, 64, 1, 8, 2, 0.0, False), (128, 256, 8, 32, 128, 0.0, False),
    (255, 9, 4, 3, None, 0.1, True), (256, 1024, 4, 16, None, 0.0, False), (1023, 2, 1, 1, None, 0.0, False),
    (512, 2, 2, 2, None, 0.0, False), (1025, 300, 4, 4, 8, 0.05, False), (2048, 128, 2, 8, 16, 0.0, False),
    (4097, 64, 1, 1, None, 0.3, True), (1500, 33, 3, 3, None, 0.0, True), (3000, 512, 8, 64, 40, 0.0, False),
    (9000, 1024, 32, 8, None, 0.01, False), (20001, 96, 6, 12, 1200, 0.0, False), (700, 1, 1, 1, 500, 0.0, False),
]


@pytest.mark.parametrize("T,E,k,P,cap,mask,dup", LAYOUT_FUZZ)
def test_layout_fuzz(T, E, k, P, cap, mask, dup):
    rng = np.random.default_rng(T * 7919 + E * 31 + k)
    if dup:
        idx = rng.integers(0, E, size=(T, k))
    else:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k]
    idx = idx.astype(np.int32)
    idx[rng.random((T, k)) < mask] = -1
    wl = W.Workload("fuzz", T=T, H=8, E=E, k=k, P=P, routing="uniform", fp8=False,
                    mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
    assert_layout_equal(gpu_layout(plan_for(wl), idx), oracle_layout(wl, idx))


def test_layout_all_copies_to_one_expert_and_overflow():
    T, E, k = 5000, 64, 1
    idx = np.full((T, k), 37, np.int32)
    for cap in (None, 100):
        wl = W.Workload("one", T=T, H=8, E=E, k=k, P=8, routing="uniform", fp8=False,
                        mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
        g = gpu_layout(plan_for(wl), idx)
        o = oracle_layout(wl, idx)
        assert_layout_equal(g, o)
        assert bool(g["err"] & ep.ERRF_CAPACITY) == (cap is not None)


def test_layout_bad_ids_flagged():
    idx = np.array([[0, 16], [-7, 3], [15, -1], [2, 99]], np.int32)
    wl = W.Workload("bad", T=4, H=8, E=16, k=2, P=4, routing="uniform", fp8=False)
    g = gpu_layout(plan_for(wl), idx)
    assert_layout_equal(g, oracle_layout(wl, idx))
    assert g["err"] == ep.ERRF_BAD_EXPERT
    big = np.random.default_rng(0).integers(-3, 20, size=(6000, 2)).astype(np.int32)
    wl = W.Workload("bad2", T=6000, H=8, E=16, k=2, P=1, routing="uniform", fp8=False)
    assert_layout_equal(gpu_layout(plan_for(wl), big), oracle_layout(wl, big))


def test_layout_empty():
    for cap in (None, 3):
        wl = W.Workload("empty", T=0, H=8, E=8, k=2, P=2, routing="uniform", fp8=False,
                        mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
        idx = np.zeros((0, 2), np.int32)
        assert_layout_equal(gpu_layout(plan_for(wl), idx), oracle_layout(wl, idx))


def test_layout_is_deterministic_and_on_any_stream():
    d = W.make("skewed")
    wl = d["wl"]
    plan = plan_for(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = gpu_layout(plan, d["topk_idx"])
    b = gpu_layout(plan, d["topk_idx"])
    assert_layout_equal(a, b)


# -------------------------------------------------------------- bf16 dispatch

def _dispatch_bf16_case(wl: W.Workload, idx, x, w, sentinel=0x7FBF):
    plan = plan_for(wl, with_weights=True)
    plan.recv.view(torch.int16).fill_(sentinel)
    plan.recv_w.fill_(-1.0)
    plan.layout(dev(idx))
    recv, _, recv_w = plan.dispatch(bf16_dev(x), dev(w))
    torch.cuda.synchronize()
    L = oracle_layout(wl, idx)
    o_recv = np.full((wl.R, wl.H), sentinel, np.uint16)
    o_recv, o_w = oracle.dispatch_bf16(x, L["slot_of"], wl.R, w, recv=o_recv)
    live = L["slot_of"][L["slot_of"] >= 0]
    o_w_full = np.full(wl.R, -1.0, np.float32)
    o_w_full[live] = o_w[live]
    np.testing.assert_array_equal(bits(recv), o_recv)
    np.testing.assert_array_equal(recv_w.cpu().numpy(), o_w_full)
    assert int(plan.layout_out.err_flags.item()) & ep.ERRF_TIMEOUT == 0


@pytest.mark.parametrize("name,T", [("tiny", None), ("prefill", None), ("grouped", 1536), ("prefill", 7)])
def test_dispatch_bf16_workloads(name, T):
    wl = W.WORKLOADS[name] if T is None else W.WORKLOADS[name].shrink(T)
    d = W.make(wl)
    _dispatch_bf16_case(wl, d["topk_idx"], d["x"], d["topk_w"])


@pytest.mark.parametrize("T,H,E,k,cap", [(1, 8, 4, 1, None), (3, 24, 4, 4, None), (200, 1032, 32, 6, None),
                                         (17, 4104, 16, 3, 2), (64, 7168, 256, 8, 4), (1, 16384, 8, 8, None),
                                         (5, 65536, 4, 2, None), (300, 136, 8, 8, None)])
def test_dispatch_bf16_shapes(T, H, E, k, cap):
    rng = np.random.default_rng(T + H)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < 0.1] = -1
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    w = rng.random((T, k)).astype(np.float32)
    wl = W.Workload("s", T=T, H=H, E=E, k=k, P=1, routing="uniform", fp8=False,
                    mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
    _dispatch_bf16_case(wl, idx, x, w)


def test_dispatch_bf16_full_size_grouped():
    """Full group-limited size (T = 16384, H = 4096, 131072 receive rows):
    layout and the whole receive buffer against the oracle's, bit for bit."""
    d = W.make("grouped")
    wl = d["wl"]
    _dispatch_bf16_case(wl, d["topk_idx"], d["x"], d["topk_w"])


# --------------------------------------------------------------- fp8 dispatch

def _dispatch_fp8_case(wl: W.Workload, idx, x):
    plan = plan_for(wl)
    plan.recv.view(torch.uint8).fill_(0x5A)
    plan.recv_scales.fill_(-3.0)
    plan.layout(dev(idx))
    q, s, _ = plan.dispatch(bf16_dev(x))
    torch.cuda.synchronize()
    L = oracle_layout(wl, idx)
    oq, os_, _ = oracle.dispatch_fp8(x, L["slot_of"], wl.R)
    live = np.zeros(wl.R, bool)
    live[L["slot_of"][L["slot_of"] >= 0]] = True
    gq = q.view(torch.uint8).cpu().numpy()
    gs = s.cpu().numpy()
    np.testing.assert_array_equal(gq[live], oq[live])
    np.testing.assert_array_equal(gs[live].view(np.uint32), os_[live].view(np.uint32))
    assert (gq[~live] == 0x5A).all() and (gs[~live] == -3.0).all()     # untouched rows
    assert int(plan.layout_out.err_flags.item()) & ep.ERRF_TIMEOUT == 0


@pytest.mark.parametrize("name,T", [("decode", None), ("skewed", 640), ("decode", 1), ("skewed", 33),
                                    ("unbalanced", None)])
def test_dispatch_fp8_workloads(name, T):
    wl = W.WORKLOADS[name] if T is None else W.WORKLOADS[name].shrink(T)
    d = W.make(wl)
    _dispatch_fp8_case(wl, d["topk_idx"], d["x"])


@pytest.mark.parametrize("T,H,E,k", [(1, 128, 4, 1), (9, 384, 8, 3), (70, 512, 16, 8), (5, 7168, 32, 8),
                                     (300, 1024, 64, 4), (2, 65536, 4, 2), (160, 640, 8, 8)])
def test_dispatch_fp8_shapes(T, H, E, k):
    rng = np.random.default_rng(T * 3 + H)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < 0.1] = -1
    scale = np.exp(rng.uniform(-20, 12, size=(T, H // 128, 1))).astype(np.float32)
    xf = (rng.standard_normal((T, H // 128, 128)).astype(np.float32) * scale).reshape(T, H)
    xf[:, :128] = 0.0                                        # an all-zero block per token
    if H >= 384:
        xf[:, 256:384] = np.float32(1e-30)                   # amax under the 1e-4 floor
    x = W.to_bf16_bits(xf)
    wl = W.Workload("s", T=T, H=H, E=E, k=k, P=1, routing="uniform", fp8=True)
    _dispatch_fp8_case(wl, idx, x)


def test_dispatch_fp8_full_size_skewed():
    """Full skewed size (T = 8192, Zipf routing, 65536 receive rows): every
    code and scale of the receive buffer against the oracle's, bit for bit."""
    d = W.make("skewed")
    wl = d["wl"]
    _dispatch_fp8_case(wl, d["topk_idx"], d["x"])


def test_dispatch_fp8_ue8m0_full_size_skewed():
    """The same full skewed dispatch with power-of-two (UE8M0) scales: every
    code and exponent byte against the oracle's."""
    d = W.make("skewed")
    wl = d["wl"]
    plan = ep.Plan(wl.T, wl.H, wl.E, wl.k, wl.P, None, fp8=True, scale_fmt="ue8m0")
    plan.layout(dev(d["topk_idx"]))
    q, e, _ = plan.dispatch(bf16_dev(d["x"]))
    torch.cuda.synchronize()
    assert int(plan.layout_out.err_flags.item()) == 0
    L = oracle_layout(wl, d["topk_idx"])
    assert (L["slot_of"] >= 0).all()           # packed, nothing masked: every row holds a copy
    oq, oe, _ = oracle.dispatch_fp8_ue8m0(d["x"], L["slot_of"], wl.R)
    np.testing.assert_array_equal(q.view(torch.uint8).cpu().numpy(), oq)
    np.testing.assert_array_equal(e.cpu().numpy(), oe)


# -------------------------------------------------------------------- combine

def _combine_case(wl: W.Workload, idx, w, y_bits):
    plan = plan_for(wl)
    plan.layout(dev(idx))
    out = plan.combine(bf16_dev(y_bits), dev(w))
    torch.cuda.synchronize()
    L = oracle_layout(wl, idx)
    assert_combine_close(bits(out), oracle.combine(y_bits, w, L["slot_of"]))


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("prefill", None), ("skewed", None),
                                    ("grouped", None), ("unbalanced", None), ("skewed", 512), ("grouped", 1024),
                                    ("tiny", 1)])
def test_combine_workloads(name, T):
    """Every workload at full size (and shrunken), whole output against the oracle."""
    wl = W.WORKLOADS[name] if T is None else W.WORKLOADS[name].shrink(T)
    d = W.make(wl)
    y = W.expert_rows(wl.R, wl.H)
    _combine_case(wl, d["topk_idx"], d["topk_w"], y)


def test_combine_random_scale_experts_tiny():
    """y = bf16(s_e * x[src]) for each receive row (fake experts with a scale each)."""
    d = W.make("tiny")
    wl = d["wl"]
    L = oracle_layout(wl, d["topk_idx"])
    s_e = W.expert_scales(wl)
    expert_of_row = np.repeat(np.arange(wl.E), L["counts"])
    xf = oracle.bf16_to_f32(d["x"])
    y = W.to_bf16_bits(xf[L["src_token"]] * s_e[expert_of_row][:, None])
    _combine_case(wl, d["topk_idx"], d["topk_w"], y)


@pytest.mark.parametrize("T,H,E,k,cap,mask", [(1, 8, 2, 1, None, 0.0), (3, 16, 4, 4, None, 0.5),
                                              (129, 1032, 16, 5, None, 0.1), (40, 7168, 64, 8, 2, 0.0),
                                              (7, 24, 32, 32, None, 0.2), (2, 65536, 8, 3, None, 0.0)])
def test_combine_shapes(T, H, E, k, cap, mask):
    rng = np.random.default_rng(T * 11 + H)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < mask] = -1
    w = rng.standard_normal((T, k)).astype(np.float32)
    wl = W.Workload("s", T=T, H=H, E=E, k=k, P=1, routing="uniform", fp8=False,
                    mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
    y = W.to_bf16_bits((rng.standard_normal((wl.R, H)) * 4).astype(np.float32))
    _combine_case(wl, idx, w, y)


# Batch sizes on both sides of the slicing steps (a row cut into 4, 2 or 1
# slices at 1024 channels, top-4) and of the switch from one resident CTA per
# unit to the persistent ring (7168 channels, top-8: 7 slices a row, about 152
# tokens' worth of units resident at once).
@pytest.mark.parametrize("T,H,E,k", [(151, 1024, 16, 4), (152, 1024, 16, 4), (305, 1024, 16, 4),
                                     (152, 7168, 256, 8), (153, 7168, 256, 8)])
def test_combine_around_the_slicing_steps(T, H, E, k):
    rng = np.random.default_rng(T * 3 + k)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    w = rng.standard_normal((T, k)).astype(np.float32)
    wl = W.Workload("s", T=T, H=H, E=E, k=k, P=1, routing="uniform", fp8=False, mode=W.PACKED, capacity=0)
    y = W.to_bf16_bits((rng.standard_normal((wl.R, H)) * 4).astype(np.float32))
    _combine_case(wl, idx, w, y)


@pytest.mark.parametrize("name", ["tiny", "prefill", "grouped"])
def test_round_trip_identity_experts_full_size(name):
    """combine(dispatch(x)) with softmax weights returns x (sum of weights ~ 1)."""
    d = W.make(name)
    wl = d["wl"]
    plan = plan_for(wl)
    x = bf16_dev(d["x"])
    plan.layout(dev(d["topk_idx"]))
    recv, _, _ = plan.dispatch(x)
    out = plan.combine(recv, dev(d["topk_w"])).float()
    xf = x.float()
    assert bool(((out - xf).abs() <= ATOL + RTOL * xf.abs()).all())


def test_out_of_range_slots_are_skipped_and_flagged():
    """slot_of entries outside [-1, R) never reach memory: skipped, EP_ERRF_BAD_SLOT set."""
    T, H, E, k = 6, 256, 4, 2
    rng = np.random.default_rng(9)
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    for fp8 in (False, True):
        plan = ep.Plan(T, H, E, k, fp8=fp8)
        slot = np.arange(T * k, dtype=np.int32).reshape(T, k)
        slot[1, 0] = plan.R + 5
        slot[4, 1] = -3
        sentinel = 0x11
        plan.recv.view(torch.uint8).fill_(sentinel)
        plan.layout_out.err_flags.zero_()
        recv, _, _ = plan.dispatch(bf16_dev(x), slot_of=dev(slot))
        torch.cuda.synchronize()
        assert int(plan.layout_out.err_flags.item()) == ep.ERRF_BAD_SLOT
        raw = recv.view(torch.uint8).cpu().numpy()
        assert (raw[2 * 1 + 0] == sentinel).all() and (raw[4 * 2 + 1] == sentinel).all()
        assert not (raw[0] == sentinel).all()
    plan = ep.Plan(T, H, E, k)
    plan.layout_out.err_flags.zero_()
    y = W.to_bf16_bits(rng.standard_normal((plan.R, H)).astype(np.float32))
    w = np.ones((T, k), np.float32)
    out = plan.combine(bf16_dev(y), dev(w), slot_of=dev(slot))
    torch.cuda.synchronize()
    assert int(plan.layout_out.err_flags.item()) == ep.ERRF_BAD_SLOT
    o = oracle.combine(y, w, np.where((slot >= 0) & (slot < plan.R), slot, -1).astype(np.int32))
    assert_combine_close(bits(out), o)


# ------------------------------------------------- fused layout + dispatch

FUSED_CASES = [
    # (T, H, E, k, P, capacity or None, fp8, mask_frac, duplicates)
    (128, 7168, 256, 8, 32, 128, True, 0.0, False),      # decode-shaped
    (128, 1024, 16, 4, 1, None, False, 0.0, False),      # tiny-shaped
    (1, 128, 4, 1, 1, None, True, 0.0, False),
    (3, 8, 4, 4, 2, 1, False, 0.2, True),                # capacity overflow, masks, duplicates
    (200, 384, 64, 6, 8, None, True, 0.1, False),        # fp8 scales stored per element
    (64, 4104, 1024, 32, 16, None, False, 0.0, False),   # k = 32, E = 1024, odd row size
    (256, 7168, 256, 8, 32, None, True, 0.0, False),     # N = 2048, the fused limit
    (300, 7168, 256, 8, 32, None, True, 0.0, False),     # beyond it: the two-call path
    (17, 2048, 32, 8, 4, 3, False, 0.05, True),
    (60, 1024, 64, 32, 4, None, True, 0.05, False),      # fp8, k = 32: four passes of eight copies
    (96, 2048, 128, 16, 8, 8, True, 0.0, True),          # fp8 into a capacity buffer that overflows
    (2048, 256, 64, 1, 4, None, False, 0.05, False),     # T = 2048 (the fused limit), k = 1: more units than SMs
    (2048, 768, 32, 1, 2, 64, True, 0.0, False),         # the same with fp8 (6 blocks, one chunk) and capacity drops
    (80, 7680, 1024, 3, 8, None, True, 0.0, True),       # fp8, 60 blocks per row: five full chunks of 12
]


@pytest.mark.parametrize("T,H,E,k,P,cap,fp8,mask,dup", FUSED_CASES)
def test_layout_dispatch_matches_oracle(T, H, E, k, P, cap, fp8, mask, dup):
    rng = np.random.default_rng(T * 13 + H + E)
    if dup:
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    else:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < mask] = -1
    if T >= 3:
        idx[1, 0] = E + 3                                    # a bad id: flagged, treated as masked
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32) * 2)
    w = rng.random((T, k)).astype(np.float32)
    wl = W.Workload("f", T=T, H=H, E=E, k=k, P=P, routing="uniform", fp8=fp8,
                    mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
    plan = plan_for(wl, with_weights=True)
    plan.recv.view(torch.uint8).fill_(0x33)
    plan.recv_w.fill_(-1.0)
    L, recv, scales, recv_w = plan.layout_dispatch(dev(idx), bf16_dev(x), dev(w))
    torch.cuda.synchronize()
    g = {key: getattr(L, key).cpu().numpy() for key in
         ("counts", "offsets", "part_counts", "part_offsets", "slot_of", "src_token", "src_k")}
    g["err"] = int(L.err_flags.cpu().numpy().view(np.uint32)[0])
    o = oracle_layout(wl, idx)
    assert_layout_equal(g, o)
    live = np.zeros(wl.R, bool)
    live[o["slot_of"][o["slot_of"] >= 0]] = True
    raw = recv.view(torch.uint8).cpu().numpy().reshape(wl.R, -1)
    if fp8:
        oq, os_, ow = oracle.dispatch_fp8(x, o["slot_of"], wl.R, w)
        np.testing.assert_array_equal(raw[live], oq[live])
        np.testing.assert_array_equal(scales.cpu().numpy()[live].view(np.uint32), os_[live].view(np.uint32))
    else:
        orecv, ow = oracle.dispatch_bf16(x, o["slot_of"], wl.R, w)
        np.testing.assert_array_equal(raw[live].view(np.uint16), orecv[live])
    assert (raw[~live] == 0x33).all()
    np.testing.assert_array_equal(recv_w.cpu().numpy()[live], ow[live])
    assert (recv_w.cpu().numpy()[~live] == -1.0).all()


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_layout_dispatch_workloads_equal_separate_calls(name):
    d = W.make(name)
    wl = d["wl"]
    a, b = plan_for(wl), plan_for(wl)
    La, ra, sa, _ = a.layout_dispatch(dev(d["topk_idx"]), bf16_dev(d["x"]))
    Lb = b.layout(dev(d["topk_idx"]))
    rb, sb, _ = b.dispatch(bf16_dev(d["x"]))
    torch.cuda.synchronize()
    for key in ("counts", "offsets", "part_counts", "part_offsets", "slot_of", "src_token", "src_k", "err_flags"):
        assert torch.equal(getattr(La, key), getattr(Lb, key)), key
    live = La.slot_of.flatten().long()
    assert torch.equal(ra.view(torch.uint8)[live], rb.view(torch.uint8)[live])
    if sa is not None:
        assert torch.equal(sa[live], sb[live])


# ------------------------------------------------------------ UE8M0 scales

@pytest.mark.parametrize("T,H,E,k,cap,fused", [(128, 7168, 256, 8, 128, True), (128, 7168, 256, 8, 128, False),
                                               (640, 7168, 256, 8, None, False), (9, 384, 8, 3, None, True),
                                               (70, 512, 16, 8, None, False), (2, 65536, 4, 2, None, False)])
def test_dispatch_fp8_ue8m0_matches_oracle(T, H, E, k, cap, fused):
    rng = np.random.default_rng(T + H + 5)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < 0.05] = -1
    scale = np.exp(rng.uniform(-20, 12, size=(T, H // 128, 1))).astype(np.float32)
    xf = (rng.standard_normal((T, H // 128, 128)).astype(np.float32) * scale).reshape(T, H)
    xf[:, :128] = 0.0
    x = W.to_bf16_bits(xf)
    wl = W.Workload("u", T=T, H=H, E=E, k=k, P=1, routing="uniform", fp8=True,
                    mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
    plan = ep.Plan(T, H, E, k, 1, cap, fp8=True, scale_fmt="ue8m0")
    plan.recv.view(torch.uint8).fill_(0x5A)
    plan.recv_scales.fill_(0xEE)
    if fused:
        _, q, e, _ = plan.layout_dispatch(dev(idx), bf16_dev(x))
    else:
        plan.layout(dev(idx))
        q, e, _ = plan.dispatch(bf16_dev(x))
    torch.cuda.synchronize()
    L = oracle_layout(wl, idx)
    oq, oe, _ = oracle.dispatch_fp8_ue8m0(x, L["slot_of"], wl.R)
    live = np.zeros(wl.R, bool)
    live[L["slot_of"][L["slot_of"] >= 0]] = True
    gq = q.view(torch.uint8).cpu().numpy()
    ge = e.cpu().numpy()
    np.testing.assert_array_equal(gq[live], oq[live])
    np.testing.assert_array_equal(ge[live], oe[live])
    assert (gq[~live] == 0x5A).all() and (ge[~live] == 0xEE).all()


# ------------------------------------- expert-side weights (unweighted combine)

@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_combine_unweighted_matches_oracle_with_unit_weights(name):
    d = W.make(name)
    wl = d["wl"]
    y = W.expert_rows(wl.R, wl.H)
    plan = plan_for(wl)
    plan.layout(dev(d["topk_idx"]))
    out = plan.combine(bf16_dev(y), None)
    torch.cuda.synchronize()
    L = oracle_layout(wl, d["topk_idx"])
    ones = np.ones((wl.T, wl.k), np.float32)
    assert_combine_close(bits(out), oracle.combine(y, ones, L["slot_of"]))


def test_expert_side_weights_round_trip():
    """dispatch routes recv_w; experts scale rows by it; unweighted combine ~ weighted combine."""
    d = W.make("tiny")
    wl = d["wl"]
    plan = plan_for(wl, with_weights=True)
    plan.layout(dev(d["topk_idx"]))
    recv, _, recv_w = plan.dispatch(bf16_dev(d["x"]), dev(d["topk_w"]))
    y_weighted = (recv.float() * recv_w[:, None]).to(torch.bfloat16)
    a = plan.combine(y_weighted, None).float().clone()
    b = plan.combine(recv, dev(d["topk_w"])).float()
    assert bool(((a - b).abs() <= ATOL + RTOL * b.abs()).all())


# ------------------------------------------------- combine of fp8 expert outputs

def _fp8_expert_outputs(rng, R, H, ue8m0):
    q = rng.integers(0, 256, size=(R, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A                                   # no NaN codes
    if ue8m0:
        s = rng.integers(100, 140, size=(R, H // 128)).astype(np.uint8)
    else:
        s = np.exp(rng.uniform(-8, 8, size=(R, H // 128))).astype(np.float32)
    return q, s


def test_combine_fp8_full_size_skewed():
    """The fp8 combine in the configuration the benchmark times it in: the
    skewed workload at full size (65536 rows of 7168 e4m3 codes with f32
    block scales, 8192 tokens, top-8), every token against the oracle."""
    d = W.make("skewed")
    wl = d["wl"]
    rng = np.random.default_rng(23)
    q = rng.integers(0, 256, size=(wl.R, wl.H), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A                                   # no NaN codes
    s = np.exp(rng.uniform(-8, 8, size=(wl.R, wl.H // 128))).astype(np.float32)
    plan = plan_for(wl)
    plan.layout(dev(d["topk_idx"]))
    out = plan.combine_fp8(dev(q).view(torch.float8_e4m3fn), dev(s), dev(d["topk_w"]))
    torch.cuda.synchronize()
    assert int(plan.layout_out.err_flags.item()) == 0
    L = oracle_layout(wl, d["topk_idx"])
    assert_combine_close(bits(out), oracle.combine_fp8(q, s, d["topk_w"], L["slot_of"]))


@pytest.mark.parametrize("T,H,E,k,cap,ue8m0,weighted", [
    (128, 7168, 256, 8, 128, False, True), (128, 7168, 256, 8, 128, True, True), (1, 128, 4, 1, None, False, True),
    (9, 384, 8, 3, None, True, False), (200, 1024, 16, 8, None, False, True), (5, 65536, 4, 2, None, True, True),
    (640, 7168, 256, 8, None, False, True),
    # around the fp8 slicing steps (7 or 4 slices a row) and the switch to the ring
    (151, 7168, 256, 8, None, False, True), (152, 7168, 256, 8, None, True, True), (300, 7168, 256, 8, None, False, True),
    # top-32: 32 staged rows a unit (the one-unit kernel's limit), then the ring
    (48, 2048, 64, 32, None, False, True), (48, 2048, 64, 32, None, True, False), (700, 1024, 64, 32, None, False, True)])
def test_combine_fp8_matches_oracle(T, H, E, k, cap, ue8m0, weighted):
    rng = np.random.default_rng(T + H + 31 * ue8m0)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    idx[rng.random((T, k)) < 0.05] = -1
    wl = W.Workload("c8", T=T, H=H, E=E, k=k, P=1, routing="uniform", fp8=True,
                    mode=W.CAPACITY if cap else W.PACKED, capacity=cap or 0)
    q, s = _fp8_expert_outputs(rng, wl.R, H, ue8m0)
    w = rng.standard_normal((T, k)).astype(np.float32) if weighted else None
    plan = plan_for(wl)
    plan.layout(dev(idx))
    out = plan.combine_fp8(dev(q).view(torch.float8_e4m3fn), dev(s), None if w is None else dev(w))
    torch.cuda.synchronize()
    L = oracle_layout(wl, idx)
    assert_combine_close(bits(out), oracle.combine_fp8(q, s, w, L["slot_of"]))


def test_fp8_dispatch_then_fp8_combine_round_trip_decode():
    """GPU fp8 dispatch into the capacity buffer, identity experts, GPU fp8 combine ~ x."""
    d = W.make("decode")
    wl = d["wl"]
    plan = plan_for(wl)
    x = bf16_dev(d["x"])
    L, q, s, _ = plan.layout_dispatch(dev(d["topk_idx"]), x)
    w = torch.full((wl.T, wl.k), 1.0 / wl.k, device="cuda")
    out = plan.combine_fp8(q, s, w).float()
    xf = x.float()
    sb = s[L.slot_of[:, 0].long()].repeat_interleave(128, dim=1)
    bound = torch.maximum(2.0 ** -4 * xf.abs(), 2.0 ** -10 * sb) * 1.0001 + 2.0 ** -8 * xf.abs() + 1e-30
    assert bool(((out - xf).abs() <= bound).all())
