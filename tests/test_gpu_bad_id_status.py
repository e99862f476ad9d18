"""Bad ids through the C ABI with no counter: the call itself returns
Q2K_ERR_BAD_ID, as the pages' gather and routed calls fail for an id out of
range (mlx-native page "tests/deepseek_q2_k.rs", test
q2_k_embedding_gather_matches_canonical_rows_and_rejects_bad_ids; fn
run_expert).  The rows of bad ids are zeros, the others are the oracle's."""

import ctypes

import numpy as np
import pytest

import oracle
import q2k_workloads as wl

torch = pytest.importorskip("torch")
import ggml_q2_quantized_gb300 as q2k  # noqa: E402
from ggml_q2_quantized_gb300 import build as q2k_build  # noqa: E402

pytestmark = pytest.mark.gpu

OK, INVALID, BAD_ID = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    q2k_build.build()
    lib = q2k.load()
    yield lib
    assert q2k.device_error() == 0, "a kernel gave up waiting on a barrier"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def stream():
    return torch.cuda.current_stream().cuda_stream


def gather_call(lib, table, ids, dim, vocab, s=None):
    out = torch.full((ids.numel(), dim), float("nan"), device="cuda")
    p = q2k.EmbeddingParams(vocab, dim, ids.numel(), 10)
    st = lib.q2k_embedding_gather(table.data_ptr(), table.numel(), ids.data_ptr(), out.data_ptr(),
                                  out.numel(), ctypes.byref(p), None,
                                  stream() if s is None else s)
    return st, out


def test_gather_null_counter_returns_bad_id(lib):
    table_np = np.concatenate([wl.page_block(r + 2) for r in range(3)])
    table = dev(table_np)
    st, out = gather_call(lib, table, dev(np.array([2, 0], dtype=np.int32)), 256, 3)
    assert st == OK, lib.q2k_last_error().decode()
    assert np.array_equal(out.cpu().numpy().view(np.uint32),
                          oracle.gather(table_np, 3, 256, [2, 0]).view(np.uint32))
    st, out = gather_call(lib, table, dev(np.array([2, 3, 7, 1], dtype=np.int32)), 256, 3)
    assert st == BAD_ID
    assert "2 id(s) out of range" in lib.q2k_last_error().decode()
    host = out.cpu().numpy()
    assert (host[1] == 0).all() and (host[2] == 0).all()
    assert np.array_equal(host[0], oracle.dequant_block(wl.page_block(4)))
    assert np.array_equal(host[3], oracle.dequant_block(wl.page_block(3)))
    # the next call with good ids is fine again (the status word starts at zero)
    st, _ = gather_call(lib, table, dev(np.array([1], dtype=np.int32)), 256, 3)
    assert st == OK


def test_gather_null_counter_refused_during_capture(lib):
    table = dev(np.concatenate([wl.page_block(r + 2) for r in range(3)]))
    ids = dev(np.array([1], dtype=np.int32))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        st, _ = gather_call(lib, table, ids, 256, 3, s=s.cuda_stream)
        g.capture_end()
    assert st == INVALID
    assert "captured" in lib.q2k_last_error().decode()


def _routed_inputs():
    rng = np.random.default_rng(77)
    n, k, experts, tokens, top_k = 40, 512, 3, 2, 2
    w = wl.random_blocks(rng, experts * n * (k // 256))
    x = rng.standard_normal((tokens, k)).astype(np.float32)
    return x, w, n, k, experts, tokens, top_k


@pytest.mark.parametrize("path", [q2k.PATH_GEMV, q2k.PATH_TENSOR])
def test_routed_null_counter_returns_bad_id(lib, path):
    x, w, n, k, experts, tokens, top_k = _routed_inputs()
    p = q2k.MatmulIdParams(tokens, top_k, n, k, experts, 10, n * (k // 256) * 84)
    ws_bytes = lib.q2k_matmul_id_workspace_bytes(path, 0, ctypes.byref(p))
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    xd, wd = dev(x), dev(w)
    for ids_np, want in ((np.array([2, 0, 1, 2], np.uint32), OK),
                         (np.array([2, 3, 1, 9], np.uint32), BAD_ID)):
        y = torch.full((ids_np.size, n), float("nan"), device="cuda")
        ids = dev(ids_np.view(np.int32))
        st = lib.q2k_matmul_id_ex(path, 0, xd.data_ptr(), xd.numel(), wd.data_ptr(), wd.numel(),
                                  ids.data_ptr(), y.data_ptr(), y.numel(), ctypes.byref(p), None,
                                  ws.data_ptr() if ws_bytes else None, ws_bytes, stream())
        assert st == want, lib.q2k_last_error().decode()
        host = y.cpu().numpy().astype(np.float64)
        tol = 1e-5 if path == q2k.PATH_GEMV else 8e-3
        for r, e in enumerate(ids_np):
            if e >= experts:
                assert (host[r] == 0).all()
                continue
            we = w[e * n * (k // 256) * 84:(e + 1) * n * (k // 256) * 84]
            yref, s = oracle.matmul(x[r // top_k:r // top_k + 1], we, n)
            assert (np.abs(host[r] - yref[0]) <= tol * s[0]).all()
    # the GEMV-path call without _ex takes the same contract
    ids = dev(np.array([0, 5, 1, 1], np.int32))
    y = torch.empty((4, n), device="cuda")
    st = lib.q2k_matmul_id(xd.data_ptr(), xd.numel(), wd.data_ptr(), wd.numel(), ids.data_ptr(),
                           y.data_ptr(), y.numel(), ctypes.byref(p), None, None, 0, stream())
    assert st == BAD_ID and "n_experts" in lib.q2k_last_error().decode()
