"""q2k_matmul_static_workspace: the tensor-core matmul for callers that cannot
allocate device memory when they call (inside a CUDA graph capture, behind a
plugin interface that only passes buffers, in a loop that must not touch the
allocator).  It keeps its scratch in a fixed array inside the library.

This file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test.  It builds and
loads the library itself, so it also passes when run alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest

import oracle
import q2k_workloads as wl
import ggml_q2_quantized_gb300 as q2k
from ggml_q2_quantized_gb300 import build as q2k_build

TOL_TC = 8e-3
STATIC_BYTES = 8 << 20


def _bind(lib):
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    f = lib.q2k_matmul_static_workspace
    f.argtypes = [vp, sz, vp, sz, vp, sz, ctypes.POINTER(q2k.MatmulParams), vp]
    f.restype = ctypes.c_int
    return f


def test_static_workspace_rejects_oversize_geometry():
    """Beyond the fixed scratch (ceil(m/256)*256 * k * 2 > 8 MiB): a clear error, no launch."""
    q2k_build.build()
    lib = q2k.load()
    f = _bind(lib)
    p = q2k.MatmulParams(1024, 8, 8192, 10)   # needs 16 MiB
    st = f(0x10000, 1024 * 8192, 0x10000000, 8 * 32 * 84, 0x20000000, 1024 * 8,
           ctypes.byref(p), None)
    assert st == 1
    assert "fixed scratch" in lib.q2k_last_error().decode()


@pytest.mark.gpu
def test_static_workspace_matches_workspace_entry_point_twice():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "needs a CUDA device"
    q2k_build.build()
    lib = q2k.load()
    f = _bind(lib)
    stream = torch.cuda.current_stream().cuda_stream

    # Two calls in a row with different shapes: the second reads a scratch that
    # still holds the first call's x image (the larger one), which must not matter.
    for seed, (m, n, k) in enumerate([(512, 7168, 1024), (40, 300, 512)]):
        x, w = wl.make_matmul_inputs(700 + seed, m, n, k)
        xd = torch.from_numpy(x).cuda()
        wd = torch.from_numpy(w).cuda()
        y_static = torch.full((m, n), float("nan"), device="cuda")
        p = q2k.MatmulParams(m, n, k, 10)
        st = f(xd.data_ptr(), xd.numel(), wd.data_ptr(), wd.numel(), y_static.data_ptr(),
               y_static.numel(), ctypes.byref(p), stream)
        assert st == 0, lib.q2k_last_error().decode()
        # the existing entry point, with a workspace from PyTorch
        y_ws = q2k.matmul(xd, wd, n, path="tensor")
        torch.cuda.synchronize()
        a = y_static.cpu().numpy().astype(np.float64)
        b = y_ws.cpu().numpy().astype(np.float64)
        assert not np.isnan(a).any()
        rows = np.arange(n) if n <= 512 else np.random.default_rng(seed).choice(n, 48, replace=False)
        _, s = oracle.matmul_rows(x, w, n, rows, threads=16)
        assert (np.abs(a[:, rows] - b[:, rows]) <= TOL_TC * s).all(), f"call {seed}: m={m} n={n} k={k}"
    err = ctypes.c_uint32(0)
    lib.q2k_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
    assert lib.q2k_device_error(ctypes.byref(err), None) == 0 and err.value == 0
