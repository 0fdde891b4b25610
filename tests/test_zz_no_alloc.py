"""ep_get_layout_static, the layout entry point for callers that cannot
allocate device memory where they compute the layout (code confined to a
memory budget owned by a host framework, or a latency-critical path on which
an allocation could stall the device).  Its scratch is an array built into the
library, so these calls pass only inputs and outputs.

Checked through the C ABI against ep_get_layout (caller-owned workspace) on
consecutive calls whose shapes differ, so stale scratch from the previous call
would show; the layout bar is bit-exact, as in the other layout tests.  This
file is collected last and also runs on its own in a fresh process.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import combine_ep_get_04_gb300 as ep
from combine_ep_get_04_gb300 import _lib
import workloads as W

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "part_counts", "part_offsets", "slot_of", "src_token", "src_k")


def _buffers(T, k, E, P, R):
    i32 = dict(dtype=torch.int32, device="cuda")
    out = dict(counts=torch.full((E,), -7, **i32), offsets=torch.full((E + 1,), -7, **i32),
               part_counts=torch.full((P,), -7, **i32), part_offsets=torch.full((P + 1,), -7, **i32),
               slot_of=torch.full((T, k), -7, **i32), src_token=torch.full((R,), -7, **i32),
               src_k=torch.full((R,), -7, **i32), err=torch.zeros(1, **i32))
    return out


def _static_layout(lib, shape, idx, out):
    st = lib.ep_get_layout_static(ctypes.byref(shape), idx.data_ptr(),
                                  *[out[key].data_ptr() for key in KEYS], out["err"].data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == _lib.EP_OK, lib.ep_last_error()
    torch.cuda.synchronize()
    return {key: out[key].cpu().numpy() for key in KEYS + ("err",)}


def _workspace_layout(T, E, k, P, cap, idx):
    plan = ep.Plan(T, 8, E, k, P, cap)
    L = plan.layout(idx)
    torch.cuda.synchronize()
    res = {key: getattr(L, key).cpu().numpy() for key in KEYS}
    res["err"] = L.err_flags.cpu().numpy()
    return res, plan.workspace_bytes


def _case(name):
    if name == "wide":
        # E = 1024, 200000 entries: 196 chunks x 1024 experts x 4 B = 784 KiB of scratch
        rng = np.random.default_rng(5)
        T, k, E, P = 25000, 8, 1024, 16
        idx = np.argsort(rng.random((T, 64)), axis=1)[:, :k].astype(np.int32) * 16
        idx[rng.random((T, k)) < 0.02] = -1
        return T, E, k, P, None, idx
    d = W.make(name)
    wl = d["wl"]
    return wl.T, wl.E, wl.k, wl.P, (wl.capacity if wl.mode == W.CAPACITY else None), d["topk_idx"]


def test_static_layout_matches_workspace_layout_on_consecutive_calls():
    lib = ep.load()
    for name in ("skewed", "wide", "grouped", "decode"):      # scratch shapes differ call to call
        T, E, k, P, cap, idx_np = _case(name)
        idx = torch.from_numpy(idx_np).cuda()
        expect, ws_bytes = _workspace_layout(T, E, k, P, cap, idx)
        shape = ep.make_shape(T, 8, E, k, P, cap)
        got = _static_layout(lib, shape, idx, _buffers(T, k, E, P, ep.recv_rows(shape)))
        for key in KEYS + ("err",):
            np.testing.assert_array_equal(got[key], expect[key], err_msg=f"{name}: {key}")
        if name != "decode":
            assert ws_bytes > 0          # these shapes do use the built-in scratch


def test_static_layout_twice_on_same_input_is_identical():
    lib = ep.load()
    T, E, k, P, cap, idx_np = _case("prefill")
    idx = torch.from_numpy(idx_np).cuda()
    shape = ep.make_shape(T, 8, E, k, P, cap)
    R = ep.recv_rows(shape)
    first = _static_layout(lib, shape, idx, _buffers(T, k, E, P, R))
    second = _static_layout(lib, shape, idx, _buffers(T, k, E, P, R))
    expect, _ = _workspace_layout(T, E, k, P, cap, idx)
    for key in KEYS + ("err",):
        np.testing.assert_array_equal(first[key], expect[key], err_msg=key)
        np.testing.assert_array_equal(second[key], expect[key], err_msg=key)


def test_static_layout_rejects_shapes_beyond_its_scratch():
    lib = ep.load()
    # 300 chunks x 1024 experts x 4 B = 1.17 MiB > 1 MiB: rejected on the host
    shape = ep.make_shape(300 * 1024 // 8, 8, 1024, 8, 1)
    st = lib.ep_get_layout_static(ctypes.byref(shape), *([None] * 9), None, None)
    assert st == _lib.EP_ERR_UNSUPPORTED
    assert b"scratch" in lib.ep_last_error()


def test_static_layout_survives_a_device_reset(tmp_path):
    """A process that resets the device between two calls gets the array of
    the new context, not an address cached from the destroyed one (a C++
    program of its own, so the reset does not touch this process's context)."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    lib_path = ep.library_path()
    exe = tmp_path / "static_after_reset"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                    "-I", os.path.join(root, "include"), os.path.join(here, "static_after_reset.cu"),
                    "-o", str(exe), lib_path, "-Xlinker", "-rpath=" + os.path.dirname(lib_path)],
                   check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "static layout across a reset ok" in res.stdout
