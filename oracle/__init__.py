"""CPU oracle for MoE token dispatch and combine (test infrastructure only).

The arithmetic lives in plain C (``ep_oracle.c``, single-threaded, built with
``-ffp-contract=off``); this module only builds it with gcc, loads it with
ctypes and marshals numpy arrays.  Nothing in the product package imports
this module: only the tests, the smoke check and the benchmark's CPU-baseline
leg do.  It shares no code with the CUDA path.

Functions and the passages they follow (DeepEP web pages):
  layout        -- per-expert counts and expert -> partition by integer
                   division ("Redundant atomics in internode_ll", quoted
                   dispatch excerpt); per-expert source order ("Reasons for not
                   calling NVSHMEM public APIs?", low-latency answer).
  dispatch_*    -- hidden row plus per-128-channel fp32 scales sent once per
                   routed expert ("Pipeline direct NVLink dispatch with
                   triple-buffered prefetch", Summary); UE8M0 power-of-two
                   scales ("Support UE8M0 data format", referenced from
                   "Redundant atomics in internode_ll").
  combine       -- weighted top-k reduce back to token order, fp32
                   accumulation, bf16 result (same PR, Validation table);
                   also over fp8 expert outputs with per-128-channel scales.
  combine_src   -- the same reduce with each copy found through the
                   expert-side record of where it came from (src_token,
                   src_k) and a per-row weight carried with the row (same
                   PR, Summary: routing information travels with the token).
All of them are pinned (tests/test_oracle_*.py); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libep_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

PACKED = 0
CAPACITY = 1
ERR_BAD_EXPERT = 1
ERR_CAPACITY = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into oracle/_build/libep_oracle.so (gcc)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp = ctypes.c_void_p
            lib.oracle_layout.restype = ctypes.c_int
            lib.oracle_layout.argtypes = [ctypes.c_int] * 6 + [vp] * 7 + [vp]
            lib.oracle_dispatch_bf16.restype = None
            lib.oracle_dispatch_bf16.argtypes = [ctypes.c_int] * 3 + [vp] * 5
            lib.oracle_dispatch_fp8.restype = None
            lib.oracle_dispatch_fp8.argtypes = [ctypes.c_int] * 3 + [vp] * 6
            lib.oracle_dispatch_fp8_ue8m0.restype = None
            lib.oracle_dispatch_fp8_ue8m0.argtypes = [ctypes.c_int] * 3 + [vp] * 6
            lib.oracle_combine_fp8.restype = None
            lib.oracle_combine_fp8.argtypes = [ctypes.c_int] * 3 + [vp, vp, ctypes.c_int, vp, vp, vp]
            lib.oracle_combine.restype = None
            lib.oracle_combine_src.restype = None
            lib.oracle_combine_src.argtypes = [ctypes.c_int] * 3 + [ctypes.c_long] + [vp] * 5
            lib.oracle_combine.argtypes = [ctypes.c_int] * 3 + [vp] * 4
            lib.oracle_e4m3_encode_n.restype = None
            lib.oracle_e4m3_encode_n.argtypes = [vp, vp, ctypes.c_long]
            lib.oracle_f32_to_bf16_n.restype = None
            lib.oracle_f32_to_bf16_n.argtypes = [vp, vp, ctypes.c_long]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def recv_rows(T: int, k: int, E: int, mode: int, cap: int) -> int:
    return T * k if mode == PACKED else E * cap


def layout(topk_idx: np.ndarray, E: int, P: int = 1, mode: int = PACKED, cap: int = 0) -> dict:
    """Counts, prefix offsets, partition sums, slot map and source maps."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    R = recv_rows(T, k, E, mode, cap)
    out = dict(
        counts=np.zeros(E, np.int32), offsets=np.zeros(E + 1, np.int32),
        part_counts=np.zeros(P, np.int32), part_offsets=np.zeros(P + 1, np.int32),
        slot_of=np.zeros((T, k), np.int32), src_token=np.zeros(R, np.int32),
        src_k=np.zeros(R, np.int32))
    err = np.zeros(1, np.uint32)
    rc = _load().oracle_layout(T, E, k, P, mode, cap, _ptr(idx), _ptr(out["counts"]),
                               _ptr(out["offsets"]), _ptr(out["part_counts"]),
                               _ptr(out["part_offsets"]), _ptr(out["slot_of"]),
                               _ptr(out["src_token"]), _ptr(out["src_k"]), _ptr(err))
    if rc != 0:
        raise ValueError("oracle_layout: bad arguments")
    out["err"] = int(err[0])
    return out


def dispatch_bf16(x: np.ndarray, slot_of: np.ndarray, R: int, topk_w: np.ndarray | None = None,
                  recv: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray | None]:
    """x: [T, H] uint16 (bf16 bits). Returns (recv [R, H] uint16, recv_w [R] or None)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    k = slot_of.shape[1]
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    if recv is None:
        recv = np.zeros((R, H), np.uint16)
    recv_w = None
    w = None
    if topk_w is not None:
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
        recv_w = np.zeros(R, np.float32)
    _load().oracle_dispatch_bf16(T, H, k, _ptr(x), _ptr(slot_of), _ptr(w), _ptr(recv), _ptr(recv_w))
    return recv, recv_w


def dispatch_fp8(x: np.ndarray, slot_of: np.ndarray, R: int, topk_w: np.ndarray | None = None):
    """Returns (recv_q [R, H] uint8 e4m3 codes, recv_s [R, H/128] f32, recv_w or None)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    if H % 128:
        raise ValueError("fp8 dispatch needs H % 128 == 0")
    k = slot_of.shape[1]
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    recv_q = np.zeros((R, H), np.uint8)
    recv_s = np.zeros((R, H // 128), np.float32)
    recv_w = None
    w = None
    if topk_w is not None:
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
        recv_w = np.zeros(R, np.float32)
    _load().oracle_dispatch_fp8(T, H, k, _ptr(x), _ptr(slot_of), _ptr(w), _ptr(recv_q),
                                _ptr(recv_s), _ptr(recv_w))
    return recv_q, recv_s, recv_w


def dispatch_fp8_ue8m0(x: np.ndarray, slot_of: np.ndarray, R: int, topk_w: np.ndarray | None = None):
    """Returns (recv_q [R, H] uint8 e4m3 codes, recv_e [R, H/128] uint8 biased exponents, recv_w)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    if H % 128:
        raise ValueError("fp8 dispatch needs H % 128 == 0")
    k = slot_of.shape[1]
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    recv_q = np.zeros((R, H), np.uint8)
    recv_e = np.zeros((R, H // 128), np.uint8)
    recv_w = None
    w = None
    if topk_w is not None:
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
        recv_w = np.zeros(R, np.float32)
    _load().oracle_dispatch_fp8_ue8m0(T, H, k, _ptr(x), _ptr(slot_of), _ptr(w), _ptr(recv_q), _ptr(recv_e),
                                      _ptr(recv_w))
    return recv_q, recv_e, recv_w


def ue8m0_value(e: np.ndarray) -> np.ndarray:
    """Scale values of UE8M0 exponent bytes: 2^(e - 127)."""
    return np.ldexp(1.0, np.asarray(e, dtype=np.int64) - 127)


def combine(y: np.ndarray, topk_w: np.ndarray, slot_of: np.ndarray) -> np.ndarray:
    """y: [R, H] uint16 (bf16 bits); returns out [T, H] uint16 (bf16 bits)."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    H = y.shape[1]
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, k = slot_of.shape
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine(T, H, k, _ptr(y), _ptr(w), _ptr(slot_of), _ptr(out))
    return out


def combine_fp8(yq: np.ndarray, ys: np.ndarray, topk_w: np.ndarray | None, slot_of: np.ndarray) -> np.ndarray:
    """yq: [R, H] uint8 e4m3 codes; ys: [R, H/128] float32 scales or uint8 UE8M0
    exponents; returns out [T, H] uint16 (bf16 bits)."""
    yq = np.ascontiguousarray(yq, dtype=np.uint8)
    H = yq.shape[1]
    if H % 128:
        raise ValueError("fp8 combine needs H % 128 == 0")
    ue8m0 = ys.dtype == np.uint8
    ys = np.ascontiguousarray(ys)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32)
    T, k = slot_of.shape
    w = None if topk_w is None else np.ascontiguousarray(topk_w, dtype=np.float32)
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine_fp8(T, H, k, _ptr(yq), _ptr(ys), int(ue8m0), _ptr(w), _ptr(slot_of), _ptr(out))
    return out


def combine_src(y: np.ndarray, row_w: np.ndarray | None, src_token: np.ndarray, src_k: np.ndarray,
                T: int, k: int) -> np.ndarray:
    """Combine addressed by the expert-side maps: y [R, H] uint16 (bf16 bits),
    row_w [R] float32 or None (unit weights), src_token / src_k [R] int32
    (-1 in rows without a copy); returns out [T, H] uint16 (bf16 bits)."""
    if k > 64:
        raise ValueError("combine_src takes k <= 64")
    y = np.ascontiguousarray(y, dtype=np.uint16)
    R, H = y.shape
    src_token = np.ascontiguousarray(src_token, dtype=np.int32)
    src_k = np.ascontiguousarray(src_k, dtype=np.int32)
    if src_token.shape != (R,) or src_k.shape != (R,):
        raise ValueError("src_token and src_k need one entry per row of y")
    w = None if row_w is None else np.ascontiguousarray(row_w, dtype=np.float32)
    out = np.zeros((T, H), np.uint16)
    _load().oracle_combine_src(T, H, k, R, _ptr(y), _ptr(w), _ptr(src_token), _ptr(src_k), _ptr(out))
    return out


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_n(_ptr(v), _ptr(codes), v.size)
    return codes


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def e4m3_table() -> np.ndarray:
    """Values of all 256 codes (float64; NaN for the two NaN codes)."""
    return np.array([e4m3_value(c) for c in range(256)], np.float64)


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    b = np.empty(v.shape, np.uint16)
    _load().oracle_f32_to_bf16_n(_ptr(v), _ptr(b), v.size)
    return b


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
