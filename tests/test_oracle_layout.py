"""Pins for the oracle's layout (counts, offsets, partitions, slot and source maps).

Pinned against: the hand-worked example in golden/layout_example.txt; numpy's
stable argsort (a library routine: a stable counting sort of the flattened
expert ids is exactly the packed row order); brute force over every input of a
tiny shape; and invariants that hold at any size.
"""
import itertools

import numpy as np
import pytest

import oracle
import workloads as W
from conftest import ints, read_golden_kv


def test_golden_layout_example():
    g = read_golden_kv("layout_example.txt")
    T, E, P, k = (int(g[n][0]) for n in ("T", "E", "P", "k"))
    idx = ints(g["topk_idx"]).reshape(T, k)
    L = oracle.layout(idx, E, P)
    for key in ("counts", "offsets", "part_counts", "part_offsets", "src_token", "src_k"):
        np.testing.assert_array_equal(L[key], ints(g[key]), err_msg=key)
    np.testing.assert_array_equal(L["slot_of"].ravel(), ints(g["slot_of"]))
    assert L["err"] == int(g["err"][0])

    cap = int(g["cap"][0])
    C = oracle.layout(idx, E, P, oracle.CAPACITY, cap)
    np.testing.assert_array_equal(C["slot_of"].ravel(), ints(g["cap_slot_of"]))
    np.testing.assert_array_equal(C["src_token"], ints(g["cap_src_token"]))
    np.testing.assert_array_equal(C["src_k"], ints(g["cap_src_k"]))
    assert C["err"] == int(g["cap_err"][0])
    # counts report the demand, not what fits
    np.testing.assert_array_equal(C["counts"], ints(g["counts"]))


def _check_against_argsort(idx: np.ndarray, E: int, P: int):
    """Packed layout == stable argsort of the flattened ids (masked last)."""
    T, k = idx.shape
    L = oracle.layout(idx, E, P)
    flat = idx.ravel().astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    keys = np.where(valid, flat, E)
    order = np.argsort(keys, kind="stable")
    n_live = int(valid.sum())
    src = order[:n_live]                            # flat (t, j) of each packed row
    np.testing.assert_array_equal(L["src_token"][:n_live], src // k)
    np.testing.assert_array_equal(L["src_k"][:n_live], src % k)
    assert (L["src_token"][n_live:] == -1).all() and (L["src_k"][n_live:] == -1).all()
    # slot_of is the inverse permutation on live entries, -1 elsewhere
    expect_slot = np.full(T * k, -1, np.int64)
    expect_slot[src] = np.arange(n_live)
    np.testing.assert_array_equal(L["slot_of"].ravel(), expect_slot)
    # counts / offsets / partitions from library routines
    counts = np.bincount(flat[valid], minlength=E)
    np.testing.assert_array_equal(L["counts"], counts)
    np.testing.assert_array_equal(L["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    pc = counts.reshape(P, E // P).sum(axis=1)
    np.testing.assert_array_equal(L["part_counts"], pc)
    np.testing.assert_array_equal(L["part_offsets"], np.concatenate([[0], np.cumsum(pc)]))
    return L


def _check_capacity(idx: np.ndarray, E: int, P: int, cap: int):
    """Capacity slot = e*cap + rank, rank = position among the expert's copies."""
    T, k = idx.shape
    flat = idx.ravel().astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    order = np.argsort(np.where(valid, flat, E), kind="stable")
    counts = np.bincount(flat[valid], minlength=E)
    starts = np.concatenate([[0], np.cumsum(counts)])
    expect = np.full(T * k, -1, np.int64)
    src_tok = np.full(E * cap, -1, np.int64)
    src_k = np.full(E * cap, -1, np.int64)
    dropped = False
    for pos, n in enumerate(order[: int(valid.sum())]):
        e = flat[n]
        rank = pos - starts[e]
        if rank < cap:
            expect[n] = e * cap + rank
            src_tok[e * cap + rank] = n // k
            src_k[e * cap + rank] = n % k
        else:
            dropped = True
    C = oracle.layout(idx, E, P, oracle.CAPACITY, cap)
    np.testing.assert_array_equal(C["slot_of"].ravel(), expect)
    np.testing.assert_array_equal(C["src_token"], src_tok)
    np.testing.assert_array_equal(C["src_k"], src_k)
    assert bool(C["err"] & oracle.ERR_CAPACITY) == dropped
    np.testing.assert_array_equal(C["counts"], counts)


def test_brute_force_tiny_shapes():
    """Every topk_idx in {-1..E-1}^(T*k) for tiny T, E, k; every capacity."""
    n_cases = 0
    for T, E, k in [(1, 1, 1), (2, 2, 1), (3, 2, 2), (2, 3, 2), (3, 3, 1), (2, 4, 2), (3, 3, 2)]:
        for vals in itertools.product(range(-1, E), repeat=T * k):
            idx = np.array(vals, np.int32).reshape(T, k)
            P = 2 if E % 2 == 0 else 1
            _check_against_argsort(idx, E, P)
            for cap in range(1, T * k + 1):
                _check_capacity(idx, E, P, cap)
            n_cases += 1
    assert n_cases == 2 + 9 + 729 + 256 + 64 + 625 + 4096


@pytest.mark.parametrize("T,E,k,P,mask_frac", [
    (1, 1, 1, 1, 0.0), (5, 7, 3, 1, 0.0), (64, 16, 4, 4, 0.1), (333, 256, 8, 32, 0.05),
    (1000, 128, 8, 8, 0.0), (2048, 64, 64, 8, 0.0), (17, 3, 5, 3, 0.3)])
def test_random_against_argsort(T, E, k, P, mask_frac):
    rng = np.random.default_rng(T * 131 + E)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)   # duplicates allowed
    idx[rng.random((T, k)) < mask_frac] = -1
    _check_against_argsort(idx, E, P)
    for cap in (1, 3, max(1, T // 4)):
        _check_capacity(idx, E, P, cap)


def _invariants(L, idx, E):
    T, k = idx.shape
    flat = idx.ravel()
    valid = (flat >= 0) & (flat < E)
    assert L["counts"].sum() == valid.sum()
    slots = L["slot_of"].ravel()
    live = slots[slots >= 0]
    assert len(np.unique(live)) == len(live)                     # each row used once
    t_of = np.arange(T * k) // k
    j_of = np.arange(T * k) % k
    ok = slots >= 0
    np.testing.assert_array_equal(L["src_token"][slots[ok]], t_of[ok])
    np.testing.assert_array_equal(L["src_k"][slots[ok]], j_of[ok])
    np.testing.assert_array_equal(flat[ok][np.argsort(slots[ok])],
                                  np.sort(flat[ok], kind="stable"))
    # rows of one expert are in strictly increasing (t, j) order
    for e in range(E):
        r0, r1 = L["offsets"][e], L["offsets"][e + 1]
        key = L["src_token"][r0:r1].astype(np.int64) * k + L["src_k"][r0:r1]
        assert (np.diff(key) > 0).all()


@pytest.mark.parametrize("name", ["tiny", "prefill", "skewed", "grouped"])
def test_invariants_on_workloads(name):
    d = W.make(name)
    wl = d["wl"]
    L = oracle.layout(d["topk_idx"], wl.E, wl.P)
    assert L["err"] == 0
    _invariants(L, d["topk_idx"], wl.E)


def test_decode_capacity_never_drops():
    d = W.make("decode")
    wl = d["wl"]
    C = oracle.layout(d["topk_idx"], wl.E, wl.P, oracle.CAPACITY, wl.capacity)
    assert C["err"] == 0 and (C["slot_of"] >= 0).all()
    e = d["topk_idx"].ravel()
    np.testing.assert_array_equal(C["slot_of"].ravel() // wl.capacity, e)


def test_bad_expert_ids_flagged_and_masked():
    idx = np.array([[0, 5], [-3, 1], [1, -1]], np.int32)
    L = oracle.layout(idx, 4, 1)
    assert L["err"] == oracle.ERR_BAD_EXPERT
    np.testing.assert_array_equal(L["slot_of"], [[0, -1], [-1, 1], [2, -1]])
    np.testing.assert_array_equal(L["counts"], [1, 2, 0, 0])


def test_empty_input():
    idx = np.zeros((0, 4), np.int32)
    L = oracle.layout(idx, 8, 2)
    assert L["counts"].sum() == 0 and L["offsets"][-1] == 0 and L["err"] == 0
    C = oracle.layout(idx, 8, 2, oracle.CAPACITY, 3)
    assert (C["src_token"] == -1).all() and C["src_token"].shape == (24,)


def test_bad_arguments_rejected():
    idx = np.zeros((2, 2), np.int32)
    with pytest.raises(ValueError):
        oracle.layout(idx, 6, 4)                 # E % P != 0
    with pytest.raises(ValueError):
        oracle.layout(idx, 4, 1, oracle.CAPACITY, 0)
