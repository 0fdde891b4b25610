"""The C-ABI library builds, loads and exports every symbol include/ep.h
declares; host-side argument checks reject bad calls before any CUDA call.

Runs without a GPU: only entry points that return before touching the device
are called.
"""
import ctypes
import os
import re

import pytest

import combine_ep_get_04_gb300 as ep
from combine_ep_get_04_gb300 import _lib
from combine_ep_get_04_gb300 import build as epbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    epbuild.build()
    return ep.load()


def declared_symbols() -> list[str]:
    text = open(os.path.join(ROOT, "include", "ep.h")).read()
    return re.findall(r"EP_API\s+[\w\s\*]*?\b(ep_\w+)\s*\(", text)


def test_header_declares_the_binding_names():
    assert sorted(declared_symbols()) == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # the ELF dynamic symbol table, independently of ctypes
    out = os.popen(f"nm -D --defined-only {ep.library_path()}").read()
    exported = set(re.findall(r" T (ep_\w+)", out))
    assert set(declared_symbols()) <= exported


def test_abi_version_and_status_strings(lib):
    assert lib.ep_abi_version() == 101
    assert lib.ep_status_string(0) == b"ok"
    assert lib.ep_status_string(1) == b"invalid argument"
    for st in range(5):
        assert lib.ep_status_str(st) == lib.ep_status_string(st)


def test_rows_and_workspace(lib):
    s = ep.make_shape(128, 7168, 256, 8, 32, capacity=128)
    assert ep.recv_rows(s) == 256 * 128
    assert ep.layout_workspace_bytes(s) == 0            # 1024 entries: one launch, no workspace
    s = ep.make_shape(16384, 4096, 128, 8, 8)
    assert ep.recv_rows(s) == 16384 * 8
    assert ep.layout_workspace_bytes(s) == 128 * 128 * 4  # 128 chunks x 128 experts x i32
    # combine by source maps: a [T, k] row map and a [T, k] weight map, each rounded to 256 B
    assert lib.ep_combine_src_workspace_bytes(ctypes.byref(s)) == 2 * 16384 * 8 * 4
    assert lib.ep_combine_src_workspace_bytes(ctypes.byref(ep.make_shape(3, 8, 4, 1, 1))) == 2 * 256


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(H=0), dict(H=12), dict(E=0), dict(k=0), dict(k=17), dict(num_partitions=3),
    dict(mode=2), dict(mode=1, capacity=0)])
def test_bad_shapes_rejected(lib, bad):
    f = dict(T=4, H=64, E=16, k=4, num_partitions=1, mode=0, capacity=0)
    f.update(bad)
    s = _lib.Shape(**f)
    assert lib.ep_recv_rows(ctypes.byref(s)) == -1
    st = lib.ep_get_layout(ctypes.byref(s), *([None] * 9), 0, None, None)
    assert st == _lib.EP_ERR_INVALID_ARG
    assert lib.ep_last_error()


def test_unsupported_sizes(lib):
    s = _lib.Shape(4, 64, 2048, 4, 1, 0, 0)
    assert lib.ep_dispatch(ctypes.byref(s), *([None] * 3), 0, *([None] * 5)) == _lib.EP_ERR_UNSUPPORTED
    s = _lib.Shape(4, 64, 64, 33, 1, 0, 0)
    assert lib.ep_combine(ctypes.byref(s), *([None] * 6)) == _lib.EP_ERR_UNSUPPORTED


def test_host_checks_before_device(lib):
    s = _lib.Shape(4, 64, 16, 4, 1, 0, 0)
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: rejected on the host
    # null pointers
    assert lib.ep_dispatch(ctypes.byref(s), None, None, fake, 0, fake, None, None, None, None) == 1
    # misaligned x / recv / y / out
    odd = ctypes.c_void_p(0x10002)
    assert lib.ep_dispatch(ctypes.byref(s), odd, None, fake, 0, fake, None, None, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(s), fake, None, fake, 0, odd, None, None, None, None) == 1
    assert lib.ep_combine(ctypes.byref(s), odd, fake, fake, fake, None, None) == 1
    assert lib.ep_combine(ctypes.byref(s), fake, fake, fake, odd, None, None) == 1
    # fp8 needs H % 128 == 0 and aligned scales
    assert lib.ep_dispatch(ctypes.byref(s), fake, None, fake, 1, fake, fake, None, None, None) == 1
    s128 = _lib.Shape(4, 128, 16, 4, 1, 0, 0)
    assert lib.ep_dispatch(ctypes.byref(s128), fake, None, fake, 1, fake, None, None, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(s128), fake, None, fake, 1, fake, odd, None, None, None) == 1
    # unknown payload, recv_w without topk_w
    assert lib.ep_dispatch(ctypes.byref(s), fake, None, fake, 7, fake, None, None, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(s), fake, None, fake, 0, fake, None, fake, None, None) == 1
    # layout: workspace too small for a large shape
    big = _lib.Shape(8192, 64, 16, 8, 1, 0, 0)
    assert lib.ep_get_layout(ctypes.byref(big), *([fake] * 8), None, 0, None, None) == 1
    assert b"workspace" in lib.ep_last_error()
    # combine by source maps: NULL maps, a small or misaligned workspace, a bad payload, fp8 with H % 128
    ws = lib.ep_combine_src_workspace_bytes(ctypes.byref(s))
    assert lib.ep_combine_src(ctypes.byref(s), fake, None, 0, None, None, fake, fake, fake, ws, None, None) == 1
    assert lib.ep_combine_src(ctypes.byref(s), fake, None, 0, None, fake, fake, fake, fake, ws - 4, None, None) == 1
    assert b"workspace" in lib.ep_last_error()
    assert lib.ep_combine_src(ctypes.byref(s), fake, None, 0, None, fake, fake, fake, odd, ws, None, None) == 1
    assert lib.ep_combine_src(ctypes.byref(s), fake, None, 5, None, fake, fake, fake, fake, ws, None, None) == 1
    assert lib.ep_combine_src(ctypes.byref(s), fake, fake, 1, None, fake, fake, fake, fake, ws, None, None) == 1
    assert lib.ep_combine_src(ctypes.byref(s128), fake, None, 1, None, fake, fake, fake, fake, ws, None, None) == 1
    # T == 0 is a no-op for dispatch / combine
    z = _lib.Shape(0, 64, 16, 4, 1, 0, 0)
    assert lib.ep_dispatch(ctypes.byref(z), *([None] * 3), 0, *([None] * 5)) == 0
    assert lib.ep_combine(ctypes.byref(z), *([None] * 6)) == 0
    assert lib.ep_combine_src(ctypes.byref(z), None, None, 0, *([None] * 5), 0, None, None) == 0


def test_layout_dispatch_host_checks(lib):
    """ep_layout_dispatch checks its arguments on the host, before any launch,
    on the fused path (small batches) and on the two-call path."""
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: rejected on the host
    odd = ctypes.c_void_p(0x10002)

    def call(shape, x=fake, payload=0, recv=fake, scales=None, recv_w=None, topk_w=None, idx=fake, counts=fake):
        return lib.ep_layout_dispatch(ctypes.byref(shape), idx, x, topk_w, payload, counts, fake, fake, fake,
                                      fake, fake, fake, recv, scales, recv_w, None, 0, None, None)

    small = _lib.Shape(4, 128, 16, 4, 1, 0, 0)
    assert call(small, payload=7) == _lib.EP_ERR_INVALID_ARG               # unknown payload
    assert call(small, x=None) == _lib.EP_ERR_INVALID_ARG                  # NULL x
    assert call(small, idx=None) == _lib.EP_ERR_INVALID_ARG                # NULL topk_idx
    assert call(small, counts=None) == _lib.EP_ERR_INVALID_ARG             # NULL layout output
    assert call(small, x=odd) == _lib.EP_ERR_INVALID_ARG                   # misaligned x
    assert call(small, recv=odd) == _lib.EP_ERR_INVALID_ARG                # misaligned recv
    assert call(small, payload=1) == _lib.EP_ERR_INVALID_ARG               # fp8 without scales
    assert call(small, payload=1, scales=odd) == _lib.EP_ERR_INVALID_ARG   # misaligned f32 scales
    assert call(small, recv_w=fake) == _lib.EP_ERR_INVALID_ARG             # recv_w without topk_w
    h64 = _lib.Shape(4, 64, 16, 4, 1, 0, 0)
    assert call(h64, payload=1, scales=fake) == _lib.EP_ERR_INVALID_ARG    # fp8 needs H % 128 == 0
    bad = _lib.Shape(4, 128, 16, 17, 1, 0, 0)
    assert call(bad) == _lib.EP_ERR_INVALID_ARG                            # k > E
    assert lib.ep_last_error()
    # beyond the fused limit: the two-call path rejects a short workspace
    big = _lib.Shape(8192, 128, 16, 8, 1, 0, 0)
    assert call(big) == _lib.EP_ERR_INVALID_ARG
    assert b"workspace" in lib.ep_last_error()


def test_product_path_does_not_use_the_oracle():
    """The package never imports the oracle or any CPU fallback."""
    pkg = os.path.join(ROOT, "combine_ep_get_04_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_plain_c_client_compiles_links_and_runs(tmp_path):
    """include/ep.h is a C header: a C11 program using it builds with
    warnings as errors, links against the library and passes its host-side
    checks."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    path = ep.library_path()
    exe = tmp_path / "abi_client"
    src = os.path.join(os.path.dirname(__file__), "abi_client.c")
    inc = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc, src, "-o", str(exe),
                    path, "-Wl,-rpath," + os.path.dirname(path)], check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "abi client ok" in res.stdout
