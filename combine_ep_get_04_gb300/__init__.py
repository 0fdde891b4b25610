"""Single-GPU MoE token dispatch and combine for GB300 (sm_103a).

Python face of the C ABI in include/ep.h.  PyTorch supplies device memory and
streams; every step of the work runs in the library's CUDA kernels.  This
module only checks tensors and passes their addresses.

    plan = Plan(T, H, E, k, num_partitions=P, capacity=None, fp8=False)
    plan.layout(topk_idx)           # counts, offsets, slot_of, src maps
    plan.dispatch(x, topk_w)        # recv (+ recv_scales, recv_w)
    plan.combine(y, topk_w)         # out

The operations follow the DeepEP pages: per-expert counts and expert ->
partition mapping ("Redundant atomics in internode_ll", quoted dispatch
excerpt), per-expert order ("Reasons for not calling NVSHMEM public APIs?"),
hidden rows with per-128-channel scales per routed expert and the combine that
reverses it ("Pipeline direct NVLink dispatch with triple-buffered prefetch").
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from ._lib import (CAPACITY, ERRF_BAD_EXPERT, ERRF_BAD_SLOT, ERRF_CAPACITY, ERRF_TIMEOUT, EXPORTED, MAX_EXPERTS, MAX_TOPK,
                   PACKED, PAYLOAD_BF16, PAYLOAD_FP8_E4M3, PAYLOAD_FP8_E4M3_UE8M0, EPError, Shape, check, library_path, load)

__all__ = ["Plan", "Layout", "Shape", "EPError", "get_layout", "dispatch", "combine", "load", "library_path",
           "PACKED", "CAPACITY", "PAYLOAD_BF16", "PAYLOAD_FP8_E4M3", "PAYLOAD_FP8_E4M3_UE8M0", "ERRF_BAD_EXPERT", "ERRF_CAPACITY",
           "ERRF_TIMEOUT", "ERRF_BAD_SLOT", "MAX_EXPERTS", "MAX_TOPK", "EXPORTED", "make_shape", "recv_rows",
           "layout_workspace_bytes", "fused_layout_dispatch", "FUSED_MAX_N", "FUSED_MAX_T"]


# Batches the library dispatches with the layout folded into one launch
# (same limits as the C library's fused path).
FUSED_MAX_N = 2048
FUSED_MAX_T = 2048


def fused_layout_dispatch(T: int, k: int, E: int) -> bool:
    """True when ep_layout_dispatch runs as a single kernel for this shape."""
    return 1 <= T <= FUSED_MAX_T and T * k <= FUSED_MAX_N and E <= MAX_EXPERTS


def make_shape(T: int, H: int, E: int, k: int, num_partitions: int = 1, capacity: int | None = None) -> Shape:
    mode = PACKED if capacity is None else CAPACITY
    return Shape(T, H, E, k, num_partitions, mode, capacity or 0)


def recv_rows(shape: Shape) -> int:
    r = load().ep_recv_rows(ctypes.byref(shape))
    if r < 0:
        check(1, "ep_recv_rows")
    return int(r)


def layout_workspace_bytes(shape: Shape) -> int:
    n = load().ep_layout_workspace_bytes(ctypes.byref(shape))
    if n == ctypes.c_size_t(-1).value:
        check(1, "ep_layout_workspace_bytes")
    return int(n)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "tensor",
         numel: int | None = None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr() or None


def _stream(stream: torch.cuda.Stream | None) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


@dataclass
class Layout:
    counts: torch.Tensor        # i32 [E]
    offsets: torch.Tensor       # i32 [E+1]
    part_counts: torch.Tensor   # i32 [P]
    part_offsets: torch.Tensor  # i32 [P+1]
    slot_of: torch.Tensor       # i32 [T, k]
    src_token: torch.Tensor     # i32 [R]
    src_k: torch.Tensor         # i32 [R]
    err_flags: torch.Tensor     # u32 word as i32 [1]


class Plan:
    """Pre-allocated outputs and workspace for one problem shape.

    Allocation happens here, once; layout / dispatch / combine then only
    launch kernels on the given (or current) stream.
    """

    def __init__(self, T: int, H: int, E: int, k: int, num_partitions: int = 1, capacity: int | None = None,
                 fp8: bool = False, with_weights: bool = False, device: str | torch.device = "cuda",
                 scale_fmt: str = "f32"):
        """scale_fmt (fp8 only): "f32" scales, or "ue8m0" power-of-two scales
        stored as biased exponent bytes."""
        load()
        if scale_fmt not in ("f32", "ue8m0"):
            raise ValueError(f"scale_fmt must be 'f32' or 'ue8m0', got {scale_fmt!r}")
        self.shape = make_shape(T, H, E, k, num_partitions, capacity)
        self.R = recv_rows(self.shape)
        self.fp8 = fp8
        self.scale_fmt = scale_fmt
        self.payload = (PAYLOAD_BF16 if not fp8 else
                        PAYLOAD_FP8_E4M3_UE8M0 if scale_fmt == "ue8m0" else PAYLOAD_FP8_E4M3)
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        ws = layout_workspace_bytes(self.shape)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.workspace_bytes = ws
        self.src_workspace_bytes = int(load().ep_combine_src_workspace_bytes(ctypes.byref(self.shape)))
        self.src_workspace = torch.empty(max(self.src_workspace_bytes, 1), dtype=torch.uint8, device=dev)
        self.layout_out = Layout(
            counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
            part_counts=torch.empty(num_partitions, **i32), part_offsets=torch.empty(num_partitions + 1, **i32),
            slot_of=torch.empty((T, k), **i32), src_token=torch.empty(self.R, **i32),
            src_k=torch.empty(self.R, **i32), err_flags=torch.zeros(1, **i32))
        if fp8:
            self.recv = torch.empty((self.R, H), dtype=torch.float8_e4m3fn, device=dev)
            self.recv_scales = torch.empty((self.R, H // 128), device=dev,
                                           dtype=torch.uint8 if scale_fmt == "ue8m0" else torch.float32)
        else:
            self.recv = torch.empty((self.R, H), dtype=torch.bfloat16, device=dev)
            self.recv_scales = None
        self.recv_w = torch.empty(self.R, dtype=torch.float32, device=dev) if with_weights else None
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    # -------------------------------------------------------------- calls

    def layout(self, topk_idx: torch.Tensor, stream: torch.cuda.Stream | None = None,
               clear_flags: bool = True) -> Layout:
        s = self.shape
        L = self.layout_out
        if clear_flags:
            L.err_flags.zero_()
        if tuple(topk_idx.shape) != (s.T, s.k):
            raise ValueError(f"topk_idx must be [{s.T}, {s.k}], got {tuple(topk_idx.shape)}")
        st = load().ep_get_layout(
            ctypes.byref(s), _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(L.counts), _ptr(L.offsets),
            _ptr(L.part_counts), _ptr(L.part_offsets), _ptr(L.slot_of), _ptr(L.src_token), _ptr(L.src_k),
            _ptr(self.workspace), self.workspace_bytes, _ptr(L.err_flags), _stream(stream))
        check(st, "ep_get_layout")
        return L

    def dispatch(self, x: torch.Tensor, topk_w: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None, slot_of: torch.Tensor | None = None):
        """Returns recv (and recv_scales for fp8, recv_w if requested)."""
        s = self.shape
        if tuple(x.shape) != (s.T, s.H):
            raise ValueError(f"x must be [{s.T}, {s.H}], got {tuple(x.shape)}")
        slot_of = self.layout_out.slot_of if slot_of is None else slot_of
        if self.recv_w is not None and topk_w is None:
            raise ValueError("this plan routes weights: pass topk_w")
        st = load().ep_dispatch(
            ctypes.byref(s), _ptr(x, torch.bfloat16, "x"),
            _ptr(topk_w, torch.float32, "topk_w", s.T * s.k), _ptr(slot_of, torch.int32, "slot_of", s.T * s.k),
            self.payload, _ptr(self.recv), _ptr(self.recv_scales),
            _ptr(self.recv_w) if topk_w is not None else None, _ptr(self.layout_out.err_flags), _stream(stream))
        check(st, "ep_dispatch")
        return self.recv, self.recv_scales, self.recv_w

    def layout_dispatch(self, topk_idx: torch.Tensor, x: torch.Tensor, topk_w: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None, clear_flags: bool = True):
        """layout() then dispatch() in one call (one launch for small batches).

        Returns (layout, recv, recv_scales, recv_w)."""
        s = self.shape
        L = self.layout_out
        if clear_flags:
            L.err_flags.zero_()
        if tuple(topk_idx.shape) != (s.T, s.k):
            raise ValueError(f"topk_idx must be [{s.T}, {s.k}], got {tuple(topk_idx.shape)}")
        if tuple(x.shape) != (s.T, s.H):
            raise ValueError(f"x must be [{s.T}, {s.H}], got {tuple(x.shape)}")
        if self.recv_w is not None and topk_w is None:
            raise ValueError("this plan routes weights: pass topk_w")
        st = load().ep_layout_dispatch(
            ctypes.byref(s), _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(x, torch.bfloat16, "x"),
            _ptr(topk_w, torch.float32, "topk_w", s.T * s.k), self.payload,
            _ptr(L.counts), _ptr(L.offsets), _ptr(L.part_counts), _ptr(L.part_offsets), _ptr(L.slot_of),
            _ptr(L.src_token), _ptr(L.src_k), _ptr(self.recv), _ptr(self.recv_scales),
            _ptr(self.recv_w) if topk_w is not None else None, _ptr(self.workspace), self.workspace_bytes,
            _ptr(L.err_flags), _stream(stream))
        check(st, "ep_layout_dispatch")
        return L, self.recv, self.recv_scales, self.recv_w

    def combine(self, y: torch.Tensor, topk_w: torch.Tensor | None, stream: torch.cuda.Stream | None = None,
                out: torch.Tensor | None = None, slot_of: torch.Tensor | None = None) -> torch.Tensor:
        s = self.shape
        if tuple(y.shape) != (self.R, s.H):
            raise ValueError(f"y must be [{self.R}, {s.H}], got {tuple(y.shape)}")
        out = self.out if out is None else out
        slot_of = self.layout_out.slot_of if slot_of is None else slot_of
        st = load().ep_combine(
            ctypes.byref(s), _ptr(y, torch.bfloat16, "y"), _ptr(topk_w, torch.float32, "topk_w", s.T * s.k),
            _ptr(slot_of, torch.int32, "slot_of", s.T * s.k), _ptr(out, torch.bfloat16, "out", s.T * s.H),
            _ptr(self.layout_out.err_flags), _stream(stream))
        check(st, "ep_combine")
        return out


    def combine_fp8(self, y: torch.Tensor, y_scales: torch.Tensor, topk_w: torch.Tensor | None,
                    stream: torch.cuda.Stream | None = None, out: torch.Tensor | None = None,
                    slot_of: torch.Tensor | None = None) -> torch.Tensor:
        """combine() over fp8 expert outputs: y e4m3 [R, H] and y_scales
        [R, H/128] (float32 scales, or uint8 UE8M0 exponents)."""
        s = self.shape
        if tuple(y.shape) != (self.R, s.H) or y.element_size() != 1:
            raise ValueError(f"y must be one-byte e4m3 [{self.R}, {s.H}]")
        if tuple(y_scales.shape) != (self.R, s.H // 128):
            raise ValueError(f"y_scales must be [{self.R}, {s.H // 128}]")
        if y_scales.dtype not in (torch.float32, torch.uint8):
            raise TypeError("y_scales must be float32 or uint8 (UE8M0)")
        payload = PAYLOAD_FP8_E4M3_UE8M0 if y_scales.dtype == torch.uint8 else PAYLOAD_FP8_E4M3
        out = self.out if out is None else out
        slot_of = self.layout_out.slot_of if slot_of is None else slot_of
        st = load().ep_combine_fp8(
            ctypes.byref(s), _ptr(y, None, "y"), _ptr(y_scales, None, "y_scales"), payload,
            _ptr(topk_w, torch.float32, "topk_w", s.T * s.k), _ptr(slot_of, torch.int32, "slot_of", s.T * s.k),
            _ptr(out, torch.bfloat16, "out", s.T * s.H), _ptr(self.layout_out.err_flags), _stream(stream))
        check(st, "ep_combine_fp8")
        return out


    def combine_src(self, y: torch.Tensor, row_w: torch.Tensor | None, src_token: torch.Tensor | None = None,
                    src_k: torch.Tensor | None = None, y_scales: torch.Tensor | None = None,
                    stream: torch.cuda.Stream | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
        """combine() addressed from the expert side: each row r of y is found
        through the pair (src_token[r], src_k[r]) it holds and weighted by
        row_w[r] (None: unweighted).  y is bf16 [R, H], or e4m3 [R, H] with
        y_scales [R, H/128] (float32, or uint8 UE8M0).  The maps default to
        this plan's last layout."""
        s = self.shape
        if tuple(y.shape) != (self.R, s.H):
            raise ValueError(f"y must be [{self.R}, {s.H}], got {tuple(y.shape)}")
        if y_scales is None:
            payload, ys = PAYLOAD_BF16, None
            yp = _ptr(y, torch.bfloat16, "y")
        else:
            if y.element_size() != 1 or tuple(y_scales.shape) != (self.R, s.H // 128):
                raise ValueError(f"fp8 y must be one-byte [{self.R}, {s.H}] with y_scales [{self.R}, {s.H // 128}]")
            if y_scales.dtype not in (torch.float32, torch.uint8):
                raise TypeError("y_scales must be float32 or uint8 (UE8M0)")
            payload = PAYLOAD_FP8_E4M3_UE8M0 if y_scales.dtype == torch.uint8 else PAYLOAD_FP8_E4M3
            yp, ys = _ptr(y, None, "y"), _ptr(y_scales, None, "y_scales")
        src_token = self.layout_out.src_token if src_token is None else src_token
        src_k = self.layout_out.src_k if src_k is None else src_k
        out = self.out if out is None else out
        st = load().ep_combine_src(
            ctypes.byref(s), yp, ys, payload, _ptr(row_w, torch.float32, "row_w", self.R),
            _ptr(src_token, torch.int32, "src_token", self.R), _ptr(src_k, torch.int32, "src_k", self.R),
            _ptr(out, torch.bfloat16, "out", s.T * s.H), _ptr(self.src_workspace), self.src_workspace_bytes,
            _ptr(self.layout_out.err_flags), _stream(stream))
        check(st, "ep_combine_src")
        return out


# ------------------------------------------------------- one-shot helpers

def get_layout(topk_idx: torch.Tensor, num_experts: int, num_partitions: int = 1,
               capacity: int | None = None, hidden: int = 8) -> Layout:
    T, k = topk_idx.shape
    plan = Plan(T, hidden, num_experts, k, num_partitions, capacity, device=topk_idx.device)
    return plan.layout(topk_idx)


def dispatch(x: torch.Tensor, layout: Layout, num_experts: int, k: int, capacity: int | None = None,
             fp8: bool = False, topk_w: torch.Tensor | None = None):
    T, H = x.shape
    plan = Plan(T, H, num_experts, k, layout.part_counts.numel(), capacity, fp8=fp8,
                with_weights=topk_w is not None, device=x.device)
    return plan.dispatch(x, topk_w, slot_of=layout.slot_of)


def combine(y: torch.Tensor, topk_w: torch.Tensor, slot_of: torch.Tensor, num_experts: int,
            capacity: int | None = None) -> torch.Tensor:
    T, k = slot_of.shape
    plan = Plan(T, y.shape[1], num_experts, k, 1, capacity, device=y.device)
    return plan.combine(y, topk_w, slot_of=slot_of)
