"""ctypes view of the C ABI in include/ep.h (libep_gb300.so).

Loading fails loudly if the library has not been built: there is no other
implementation behind these names.
"""
from __future__ import annotations

import ctypes
import importlib
import os

PACKED = 0
CAPACITY = 1
PAYLOAD_BF16 = 0
PAYLOAD_FP8_E4M3 = 1
PAYLOAD_FP8_E4M3_UE8M0 = 2

ERRF_BAD_EXPERT = 1
ERRF_CAPACITY = 2
ERRF_TIMEOUT = 4
ERRF_BAD_SLOT = 8

MAX_EXPERTS = 1024
MAX_TOPK = 32

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_UNSUPPORTED = 2
EP_ERR_CUDA = 3

# Every symbol include/ep.h declares.
EXPORTED = ("ep_recv_rows", "ep_layout_workspace_bytes", "ep_get_layout", "ep_get_layout_static",
            "ep_dispatch", "ep_layout_dispatch", "ep_combine", "ep_combine_fp8", "ep_combine_src_workspace_bytes",
            "ep_combine_src", "ep_status_string", "ep_status_str", "ep_last_error", "ep_abi_version")


class Shape(ctypes.Structure):
    """ep_shape_t."""
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("num_partitions", ctypes.c_int32), ("mode", ctypes.c_int32), ("capacity", ctypes.c_int32)]

    def __repr__(self) -> str:
        return (f"Shape(T={self.T}, H={self.H}, E={self.E}, k={self.k}, P={self.num_partitions}, "
                f"mode={self.mode}, capacity={self.capacity})")


class EPError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str):
        super().__init__(f"{what}: {detail or 'status ' + str(status)}")
        self.status = status


_lib = None


def library_path() -> str:
    # imported here, not at package import, so that `python -m
    # combine_ep_get_04_gb300.build` runs the module fresh
    return importlib.import_module(__package__ + ".build").LIB_PATH


def load() -> ctypes.CDLL:
    """Load libep_gb300.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first "
                          f"(python -m combine_ep_get_04_gb300.build or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, sp, i32 = ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_int32
    lib.ep_recv_rows.restype = ctypes.c_int64
    lib.ep_recv_rows.argtypes = [sp]
    lib.ep_layout_workspace_bytes.restype = ctypes.c_size_t
    lib.ep_layout_workspace_bytes.argtypes = [sp]
    lib.ep_get_layout.restype = ctypes.c_int
    lib.ep_get_layout.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
    lib.ep_get_layout_static.restype = ctypes.c_int
    lib.ep_get_layout_static.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.ep_dispatch.restype = ctypes.c_int
    lib.ep_dispatch.argtypes = [sp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
    lib.ep_layout_dispatch.restype = ctypes.c_int
    lib.ep_layout_dispatch.argtypes = [sp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                       ctypes.c_size_t, vp, vp]
    lib.ep_combine.restype = ctypes.c_int
    lib.ep_combine.argtypes = [sp, vp, vp, vp, vp, vp, vp]
    lib.ep_combine_fp8.restype = ctypes.c_int
    lib.ep_combine_fp8.argtypes = [sp, vp, vp, i32, vp, vp, vp, vp, vp]
    lib.ep_combine_src_workspace_bytes.restype = ctypes.c_size_t
    lib.ep_combine_src_workspace_bytes.argtypes = [sp]
    lib.ep_combine_src.restype = ctypes.c_int
    lib.ep_combine_src.argtypes = [sp, vp, vp, i32, vp, vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
    lib.ep_status_string.restype = ctypes.c_char_p
    lib.ep_status_string.argtypes = [ctypes.c_int]
    lib.ep_status_str.restype = ctypes.c_char_p
    lib.ep_status_str.argtypes = [ctypes.c_int]
    lib.ep_last_error.restype = ctypes.c_char_p
    lib.ep_last_error.argtypes = []
    lib.ep_abi_version.restype = ctypes.c_int32
    lib.ep_abi_version.argtypes = []
    _lib = lib
    return lib


def check(status: int, what: str) -> None:
    if status != EP_OK:
        lib = load()
        raise EPError(status, what, (lib.ep_last_error() or b"").decode())
