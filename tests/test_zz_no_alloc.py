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

# Calls in a row that all keep state in the shared array:
#   512 x 7168 x 1024  the x tile image, two 256-row super-tiles (1 MiB);
#   100 x 512 x 2048   K split in parts: the image plus the parts' partial
#                      results and the per-tile arrival counters, which must
#                      start at zero although the array holds the last call's
#                      bytes;
#   300 x 1024 x 1024  an image whose padding rows (300..511) still hold the
#                      first call's rows.
SHAPES = [(512, 7168, 1024), (100, 512, 2048), (300, 1024, 1024)]


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


def test_static_workspace_test_shapes_use_the_scratch():
    """Every shape of the GPU test needs scratch, and it fits the fixed array."""
    q2k_build.build()
    lib = q2k.load()
    for m, n, k in SHAPES:
        p = q2k.MatmulParams(m, n, k, 10)
        need = lib.q2k_matmul_workspace_bytes(ctypes.byref(p), q2k.PATH_TENSOR)
        assert 0 < need <= STATIC_BYTES, (m, n, k, need)
    # the second shape splits K: more than the x image alone
    m, n, k = SHAPES[1]
    image = -(-m // 256) * 256 * k * 2
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(q2k.MatmulParams(m, n, k, 10)),
                                          q2k.PATH_TENSOR) > image


@pytest.mark.gpu
def test_static_workspace_matches_oracle_and_workspace_entry_point():
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "needs a CUDA device"
    q2k_build.build()
    lib = q2k.load()
    f = _bind(lib)
    stream = torch.cuda.current_stream().cuda_stream

    for seed, (m, n, k) in enumerate(SHAPES):
        x, w = wl.make_matmul_inputs(700 + seed, m, n, k)
        yref, s = oracle.matmul(x, w, n, threads=16)
        xd = torch.from_numpy(x).cuda()
        wd = torch.from_numpy(w).cuda()
        # two calls in a row on the same inputs: the second starts from the
        # array the first left behind
        for rep in range(2):
            y_static = torch.full((m, n), float("nan"), device="cuda")
            p = q2k.MatmulParams(m, n, k, 10)
            st = f(xd.data_ptr(), xd.numel(), wd.data_ptr(), wd.numel(), y_static.data_ptr(),
                   y_static.numel(), ctypes.byref(p), stream)
            assert st == 0, lib.q2k_last_error().decode()
            torch.cuda.synchronize()
            a = y_static.cpu().numpy().astype(np.float64)
            assert not np.isnan(a).any()
            err = np.abs(a - yref)
            assert (err <= TOL_TC * s).all(), (
                f"m={m} n={n} k={k} call {rep}: worst err/S {(err / np.maximum(s, 1e-30)).max():.3g}")
        # the existing entry point, with a workspace from PyTorch
        y_ws = q2k.matmul(xd, wd, n, path="tensor")
        torch.cuda.synchronize()
        b = y_ws.cpu().numpy().astype(np.float64)
        assert (np.abs(a - b) <= TOL_TC * s).all(), f"static vs workspace: m={m} n={n} k={k}"
    err = ctypes.c_uint32(0)
    lib.q2k_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
    assert lib.q2k_device_error(ctypes.byref(err), None) == 0 and err.value == 0
