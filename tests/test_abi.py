"""The C ABI without a GPU: the library loads, exports every function the
header declares, lays out its structs as declared, and rejects malformed
arguments before touching CUDA (page "tests/deepseek_q2_k.rs": malformed
buffers and bad geometry are InvalidArgument, nothing is launched)."""

import ctypes
import os
import subprocess

import pytest

import ggml_q2_quantized_gb300 as q2k
from ggml_q2_quantized_gb300 import build as q2k_build

INVALID = 1


@pytest.fixture(scope="module")
def lib():
    q2k_build.build()
    return q2k.load()


def test_header_declares_the_calls():
    names = q2k.header_functions()
    for want in ("q2k_dequantize", "q2k_embedding_gather", "q2k_matmul", "q2k_matmul_path",
                 "q2k_matmul_ex", "q2k_matmul_batched_mv", "q2k_matmul_id", "q2k_device_error",
                 "q2k_last_error", "q2k_abi_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in q2k.header_functions():
        assert hasattr(lib, name), name


def test_abi_version(lib):
    assert lib.q2k_abi_version() == 1


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "q2k.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(q2k_matmul_params),"
        " offsetof(q2k_matmul_params, ggml_type), sizeof(q2k_embedding_params),"
        " offsetof(q2k_embedding_params, n_tokens), sizeof(q2k_status),"
        " sizeof(q2k_matmul_id_params), offsetof(q2k_matmul_id_params, ggml_type),"
        " offsetof(q2k_matmul_id_params, expert_stride));"
        "printf(\"%zu %zu\\n\", sizeof(q2k_gguf_tensor), offsetof(q2k_gguf_tensor, byte_len));"
        "printf(\"%zu %zu\\n\", sizeof(q2k_matmul_call), offsetof(q2k_matmul_call, flags));return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", q2k_build.INCLUDE, str(src),
                    "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert [int(v) for v in out] == [16, 12, 16, 8, 4, 32, 20, 24, 64, 56, 88, 84]
    assert ctypes.sizeof(q2k.MatmulCall) == 88 and q2k.MatmulCall.flags.offset == 84
    assert ctypes.sizeof(q2k.GgufTensor) == 64 and q2k.GgufTensor.byte_len.offset == 56
    assert ctypes.sizeof(q2k.MatmulIdParams) == 32
    assert q2k.MatmulIdParams.ggml_type.offset == 20
    assert q2k.MatmulIdParams.expert_stride.offset == 24
    assert ctypes.sizeof(q2k.MatmulParams) == 16
    assert ctypes.sizeof(q2k.EmbeddingParams) == 16
    assert q2k.MatmulParams.ggml_type.offset == 12


def _mm(lib, params, x=0x10000, xe=None, w=0x100000, wb=None, y=0x1000000, ye=None, path=0):
    m, n, k = params.m, params.n, params.k
    xe = m * k if xe is None else xe
    wb = n * (k // 256) * 84 if wb is None else wb
    ye = m * n if ye is None else ye
    return lib.q2k_matmul_path(path, x, xe, w, wb, y, ye, ctypes.byref(params), None)


P = q2k.MatmulParams


@pytest.mark.parametrize("params,kw,fragment", [
    (P(1, 8, 255, 10), {}, "multiple of 256"),
    (P(1, 8, 256, 11), {}, "not Q2_K"),
    (P(0, 8, 256, 10), {}, ">= 1"),
    (P(1, 0, 256, 10), {}, ">= 1"),
    (P(1, 8, 256, 10), {"xe": 255}, "x has 255"),
    (P(1, 8, 256, 10), {"wb": 8 * 84 - 1}, "w has 671"),
    (P(1, 8, 256, 10), {"ye": 9}, "y has 9"),
    (P(1, 8, 256, 10), {"x": 0}, "non-NULL"),
    (P(1, 8, 256, 10), {"x": 0x10004}, "aligned"),
    (P(1, 8, 256, 10), {"w": 0x100002}, "aligned"),
    (P(1, 8, 256, 10), {"y": 0x10010}, "alias"),          # y inside x
    (P(1, 8, 256, 10), {"y": 0x100000}, "alias"),         # y on top of w
    (P(1, 8, 256, 10), {"path": 7}, "unknown path"),
    (P(0xFFFFFFFF, 0xFFFFFFFF, 256, 10), {}, "signed 32-bit"),
])
def test_matmul_rejects(lib, params, kw, fragment):
    assert _mm(lib, params, **kw) == INVALID
    assert fragment in lib.q2k_last_error().decode()


def test_dequantize_rejects_malformed(lib):
    # page test q2_k_host_decode_rejects_malformed_buffers: 83 bytes, 255 floats
    assert lib.q2k_dequantize(0x10000, 83, 0x100000, 256, None) == INVALID
    assert lib.q2k_dequantize(0x10000, 84, 0x100000, 255, None) == INVALID
    assert lib.q2k_dequantize(0x10000, 0, 0x100000, 0, None) == INVALID
    assert lib.q2k_dequantize(0, 84, 0x100000, 256, None) == INVALID
    assert lib.q2k_dequantize(0x10000, 84, 0x10000, 256, None) == INVALID  # aliasing


def test_gather_rejects_malformed(lib):
    E = q2k.EmbeddingParams
    ok = dict(table=0x10000, tb=3 * 84, ids=0x20000, out=0x100000, oe=2 * 256)

    def call(p, **kw):
        a = dict(ok, **kw)
        return lib.q2k_embedding_gather(a["table"], a["tb"], a["ids"], a["out"], a["oe"],
                                        ctypes.byref(p), None, None)
    assert call(E(3, 255, 2, 10)) == INVALID
    assert call(E(3, 256, 2, 9)) == INVALID
    assert call(E(3, 256, 2, 10), tb=3 * 84 + 1) == INVALID
    assert call(E(3, 256, 2, 10), oe=511) == INVALID
    assert call(E(3, 256, 2, 10), out=0x10000) == INVALID   # out over the table
    assert call(E(0, 256, 2, 10)) == INVALID
    assert "vocab_size" in lib.q2k_last_error().decode()


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        q2k.load(str(tmp_path / "nope.so"))


def test_matmul_ex_rejects_unknown_flags(lib):
    p = q2k.MatmulParams(1, 8, 256, 10)
    assert lib.q2k_matmul_ex(0, 4, 0x10000, 256, 0x100000, 672, 0x1000000, 8,
                             ctypes.byref(p), None, 0, None) == INVALID
    assert "flag" in lib.q2k_last_error().decode()


def test_workspace_bytes(lib):
    P = q2k.MatmulParams
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(1, 8, 256, 10)), 0) == 0      # GEMV
    # m <= 64 whose K stages fit on chip: x converted in the GEMM, no workspace
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(9, 8, 256, 10)), 0) == 0
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(1, 8, 256, 10)), 2) == 0
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(16, 4096, 4096, 10)), 0) == 0
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(64, 4000, 8192, 10)), 0) == 0
    # m = 64 with 16 blocks a row and one K part: its x does not fit, x image
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(64, 14336, 4096, 10)), 0) == 256 * 4096 * 2
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(512, 7168, 7168, 10)), 0) == 512 * 7168 * 2
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(129, 8, 512, 10)), 0) == 256 * 512 * 2
    assert lib.q2k_matmul_workspace_bytes(ctypes.byref(P(9, 8, 255, 10)), 0) == 0      # invalid


def test_workspace_rejected_when_small_or_aliasing(lib):
    # m = 129 takes the x-image path, so it has a workspace to check
    p = q2k.MatmulParams(129, 8, 256, 10)
    need = 256 * 256 * 2
    args = (0x10000, 129 * 256, 0x100000, 8 * 84, 0x1000000, 129 * 8, ctypes.byref(p))
    assert lib.q2k_matmul_ex(2, 0, *args, 0x2000000, need - 1, None) == INVALID
    assert "workspace" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_ex(2, 0, *args, 0x2000008, need, None) == INVALID
    assert lib.q2k_matmul_ex(2, 0, *args, 0x10000, need, None) == INVALID   # over x


def test_selftest_wait_timeout_rejects_out_of_range_limits(lib):
    """Checked before any device work: 0 and > 100 ms are refused."""
    for bad in (0, 100001):
        assert lib.q2k_selftest_wait_timeout(bad, None) == INVALID
        assert "limit_us" in lib.q2k_last_error().decode()


def _bmv(lib, batches=3, m=1, n=8, k=256, xe=None, wb=None, ye=None, x=0x10000, w=0x100000,
         y=0x1000000):
    xe = batches * k if xe is None else xe
    wb = batches * n * (k // 256) * 84 if wb is None else wb
    ye = batches * n if ye is None else ye
    return lib.q2k_matmul_batched_mv(x, xe, w, wb, y, ye, batches, m, n, k, None, 0, None)


@pytest.mark.parametrize("kw,fragment", [
    (dict(m=2), "m = 1"),
    (dict(batches=0), "batches"),
    (dict(batches=65536), "batches"),
    (dict(k=255), "multiple of 256"),
    (dict(xe=3 * 256 - 1), "batched sizes"),
    (dict(wb=3 * 8 * 84 + 84), "batched sizes"),
    (dict(ye=3 * 8 + 1), "batched sizes"),
    (dict(x=0x10004), "aligned"),
    (dict(y=0x100000 + 112), "alias"),
])
def test_batched_mv_rejects(lib, kw, fragment):
    """Checked before any device work (the fake addresses are never touched)."""
    assert _bmv(lib, **kw) == INVALID
    assert fragment in lib.q2k_last_error().decode()


def _mid(lib, n_tokens=2, top_k=2, n=8, k=256, n_experts=3, stride=None, xe=None, wb=None,
         ye=None, ids=0x3000000, x=0x10000, w=0x100000, y=0x1000000, ggml_type=10):
    stride = n * (k // 256) * 84 if stride is None else stride
    p = q2k.MatmulIdParams(n_tokens, top_k, n, k, n_experts, ggml_type, stride)
    xe = n_tokens * k if xe is None else xe
    wb = (n_experts - 1) * stride + n * (k // 256) * 84 if wb is None else wb
    ye = n_tokens * top_k * n if ye is None else ye
    return lib.q2k_matmul_id(x, xe, w, wb, ids, y, ye, ctypes.byref(p), None, None, 0, None)


@pytest.mark.parametrize("kw,fragment", [
    (dict(ggml_type=12), "Q2_K"),
    (dict(top_k=0), ">= 1"),
    (dict(n_experts=0), ">= 1"),
    (dict(k=300), "multiple of 256"),
    (dict(stride=8 * 84 - 4), "expert_stride"),
    (dict(stride=8 * 84 + 2), "expert_stride"),
    (dict(wb=2 * 8 * 84 + 8 * 84 - 1), "w has"),
    (dict(xe=511), "x has"),
    (dict(ye=31), "y has"),
    (dict(ids=0), "non-NULL"),
    (dict(n_tokens=40000, top_k=2, xe=40000 * 256, ye=80000 * 8), "65535"),
    (dict(ids=0x1000000 + 8), "alias"),
    (dict(w=0x100002), "aligned"),
])
def test_matmul_id_rejects(lib, kw, fragment):
    assert _mid(lib, **kw) == INVALID
    assert fragment in lib.q2k_last_error().decode()


def test_matmul_id_slotted_and_pair_reject(lib):
    n_tokens, top_k, n, k, experts = 2, 2, 8, 256, 3
    p = q2k.MatmulIdParams(n_tokens, top_k, n, k, experts, 10, n * 84)
    wb = experts * n * 84
    # slotted: x holds one row per route (n_tokens*top_k*k), not per token
    assert lib.q2k_matmul_id_slotted(0x10000, n_tokens * k, 0x100000, wb, 0x3000000, 0x1000000,
                                     n_tokens * top_k * n, ctypes.byref(p), None, None, 0,
                                     None) == INVALID
    assert "n_tokens*top_k*k" in lib.q2k_last_error().decode()
    args = (0x10000, n_tokens * k, 0x100000, wb)
    # pair: missing second weight set, short second weight set, aliasing outputs
    assert lib.q2k_matmul_id_pair(*args, None, wb, 0x3000000, 0x1000000, 0x2000000,
                                  n_tokens * top_k * n, ctypes.byref(p), None, None, 0, None) == INVALID
    assert lib.q2k_matmul_id_pair(*args, 0x200000, wb - 4, 0x3000000, 0x1000000, 0x2000000,
                                  n_tokens * top_k * n, ctypes.byref(p), None, None, 0, None) == INVALID
    assert "w has" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_pair(*args, 0x200000, wb, 0x3000000, 0x1000000, 0x1000000 + 32,
                                  n_tokens * top_k * n, ctypes.byref(p), None, None, 0, None) == INVALID
    assert "alias" in lib.q2k_last_error().decode()
    big = q2k.MatmulIdParams(16384, 2, n, k, experts, 10, n * 84)
    assert lib.q2k_matmul_id_pair(0x10000, 16384 * k, 0x100000, wb, 0x200000, wb, 0x3000000,
                                  0x1000000, 0x8000000, 32768 * n, ctypes.byref(big), None,
                                  None, 0, None) == INVALID
    assert "32767" in lib.q2k_last_error().decode()


def test_matmul_id_ex_workspace_and_rejections(lib):
    """The routed product's tensor path: its workspace size (tile table, row
    routes, each route's row, x image of up to routes/128 + min(experts, routes)
    tiles) and the checks made before any device work."""
    n_tokens, top_k, n, k, experts = 64, 8, 2048, 7168, 64
    p = q2k.MatmulIdParams(n_tokens, top_k, n, k, experts, 10, n * (k // 256) * 84)
    routes = n_tokens * top_k
    tiles = routes // 128 + 64
    info = (tiles * 8 + 255) // 256 * 256
    route_rows = (routes * 4 + 255) // 256 * 256
    image = (tiles * 128 + 255) // 256 * 256 * k * 2
    want = info + tiles * 128 * 4 + route_rows + image
    assert lib.q2k_matmul_id_workspace_bytes(q2k.PATH_TENSOR, 0, ctypes.byref(p)) == want
    assert lib.q2k_matmul_id_workspace_bytes(q2k.PATH_AUTO, 0, ctypes.byref(p)) == want
    # auto takes the GEMV at <= 32 tokens: its optional scratch is the x planes
    small = q2k.MatmulIdParams(32, top_k, n, k, experts, 10, p.expert_stride)
    assert (lib.q2k_matmul_id_workspace_bytes(q2k.PATH_AUTO, 0, ctypes.byref(small))
            == lib.q2k_x_planes_bytes(k, 32))
    assert (lib.q2k_matmul_id_workspace_bytes(q2k.PATH_GEMV, q2k.ID_SLOTTED, ctypes.byref(small))
            == lib.q2k_x_planes_bytes(k, 32 * top_k))
    many = q2k.MatmulIdParams(n_tokens, top_k, n, k, 4097, 10, p.expert_stride)
    assert lib.q2k_matmul_id_workspace_bytes(q2k.PATH_TENSOR, 0, ctypes.byref(many)) == 0
    assert lib.q2k_matmul_id_workspace_bytes(q2k.PATH_TENSOR, 2, ctypes.byref(p)) == 0
    wb = experts * p.expert_stride
    args = (0x10000, n_tokens * k, 0x10000000, wb, 0x1000000, 0x200000000, 512 * n, ctypes.byref(p),
            None)
    assert lib.q2k_matmul_id_ex(7, 0, *args, None, 0, None) == INVALID
    assert "unknown path" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_ex(q2k.PATH_TENSOR, 4, *args, None, 0, None) == INVALID
    assert "flag" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_ex(q2k.PATH_TENSOR, 0, *args, None, 0, None) == INVALID
    assert "workspace" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_ex(q2k.PATH_TENSOR, 0, *args, 0x300000000, want - 16, None) == INVALID
    assert "workspace" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_ex(q2k.PATH_TENSOR, 0, *args, 0x300000008, want, None) == INVALID
    assert "aligned" in lib.q2k_last_error().decode()
    # the workspace overlapping y
    assert lib.q2k_matmul_id_ex(q2k.PATH_TENSOR, 0, *args, 0x200000000 + 4096, want, None) == INVALID
    assert "alias" in lib.q2k_last_error().decode()
    # the pair: unknown path, missing second set, workspace overlapping the second output
    pair = (0x10000, n_tokens * k, 0x10000000, wb, 0x40000000, wb, 0x1000000, 0x200000000,
            0x280000000, 512 * n, ctypes.byref(p), None)
    assert lib.q2k_matmul_id_pair_ex(9, *pair, None, 0, None) == INVALID
    assert "unknown path" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_pair_ex(q2k.PATH_TENSOR, 0x10000, n_tokens * k, 0x10000000, wb, None,
                                     wb, 0x1000000, 0x200000000, 0x280000000, 512 * n,
                                     ctypes.byref(p), None, None, 0, None) == INVALID
    assert lib.q2k_matmul_id_pair_ex(q2k.PATH_TENSOR, *pair, 0x280000000 + 64, want, None) == INVALID
    assert "alias" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_id_pair_ex(q2k.PATH_TENSOR, *pair, None, 0, None) == INVALID
    assert "workspace" in lib.q2k_last_error().decode()


def test_matmul_ex_batch_checks_every_call_first(lib):
    """A malformed call anywhere rejects the batch before any launch; its index is named."""
    calls = (q2k.MatmulCall * 2)()
    for i, c in enumerate(calls):
        c.x, c.x_elems, c.w, c.w_bytes = 0x10000, 256, 0x100000, 8 * 84
        c.y, c.y_elems = 0x1000000 + 4096 * i, 8
        c.params = q2k.MatmulParams(1, 8, 256, 10)
        c.path, c.flags = 0, 0
    calls[1].params = q2k.MatmulParams(1, 8, 255, 10)
    assert lib.q2k_matmul_ex_batch(calls, 2, None, 0, None) == INVALID
    assert "call 1:" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_batch_scratch_bytes(calls, 2) == 0
    calls[1].params = q2k.MatmulParams(1, 8, 256, 10)
    # two m = 1 calls on one x: one slot of prepared x (K/64 slices x (64 floats + 1 scale))
    assert lib.q2k_matmul_batch_scratch_bytes(calls, 2) == (4 * 260 + 255) // 256 * 256
    calls[0].flags = 8
    assert lib.q2k_matmul_ex_batch(calls, 2, None, 0, None) == INVALID
    assert "call 0:" in lib.q2k_last_error().decode()
    calls[0].flags = 0
    assert lib.q2k_matmul_ex_batch(calls, 2, 0x3000008, 2048, None) == INVALID
    assert "aligned" in lib.q2k_last_error().decode()
    # a scratch overlapping a call's output (or its x) is rejected before any launch
    assert lib.q2k_matmul_ex_batch(calls, 2, 0x1000000 + 4096, 2048, None) == INVALID
    assert "scratch must not alias call 1" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_ex_batch(calls, 2, 0x10000, 2048, None) == INVALID
    assert "scratch must not alias call 0" in lib.q2k_last_error().decode()
    assert lib.q2k_matmul_ex_batch(None, 0, None, 0, None) == 0   # nothing to do


def test_matmul_batch_plans_small_m_runs(lib):
    """The batch's runs of independent small-m tensor calls on one x (planned on
    the host, geometry only): each run gets one slot of the scratch for x's
    bf16 image (ceil(m / 256) * 256 * k * 2 bytes) when its calls have at least
    128 weight tiles of 128 rows between them; dependent calls, too few tiles,
    k not a multiple of 1024, a W that is not 16-byte aligned and a call on
    another x (which may overwrite the runs' x) all end or prevent a run."""
    m, n, k = 16, 4096, 4096
    wbytes = n * (k // 256) * 84
    image = 256 * k * 2

    def calls_for(count, flags=2, kk=k, nn=n, x=0x10000, w_off=0):
        arr = (q2k.MatmulCall * count)()
        for i, c in enumerate(arr):
            c.x, c.x_elems = x, m * kk
            c.w, c.w_bytes = 0x100000000 + i * 0x1000000 + w_off, nn * (kk // 256) * 84
            c.y, c.y_elems = 0x800000000 + i * 0x1000000, m * nn
            c.params = q2k.MatmulParams(m, nn, kk, 10)
            c.path, c.flags = q2k.PATH_TENSOR, flags
        return arr

    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(6), 6) == image      # 192 tiles: one run
    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(4), 4) == image      # 128 tiles
    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(3), 3) == 0          # 96 tiles
    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(6, flags=0), 6) == 0  # dependent
    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(6, kk=2816), 6) == 0  # k % 1024 != 0
    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(6, w_off=4), 6) == 0  # W 4-byte aligned
    assert lib.q2k_matmul_batch_scratch_bytes(calls_for(2, nn=8192), 2) == image  # 2 x 64 tiles
    # a call on another x between two runs: two slots
    arr = calls_for(9)
    arr[4].x = 0x20000
    assert lib.q2k_matmul_batch_scratch_bytes(arr, 9) == 2 * image
    # a call on another x that overwrites the runs' x: the same split
    arr = calls_for(9)
    arr[4].x, arr[4].y = 0x40000000, 0x10000
    assert lib.q2k_matmul_batch_scratch_bytes(arr, 9) == 2 * image
    # ... while the calls themselves stay as given
    assert arr[0].w_bytes == wbytes


def test_bench_launch_count_follows_the_batch_plan(lib):
    """bench.py counts a step's kernel launches from the batch's plan; for the
    workloads it times, its count agrees with the plan the library makes
    (a scratch slot per shared x conversion or small-m run)."""
    import bench

    def scratch(m, n, k, layers, flags):
        arr = (q2k.MatmulCall * layers)()
        for i, c in enumerate(arr):
            c.x, c.x_elems = 0x10000, m * k
            c.w, c.w_bytes = 0x100000000 + i * 0x4000000, n * (k // 256) * 84
            c.y, c.y_elems = 0x2000000000 + i * 0x4000000, m * n
            c.params = q2k.MatmulParams(m, n, k, 10)
            c.path, c.flags = q2k.PATH_AUTO, flags
        return lib.q2k_matmul_batch_scratch_bytes(arr, layers)

    # decode GEMV, 74 independent calls on one x: one x preparation + 74 GEMVs
    assert scratch(1, 4096, 4096, 74, 2) > 0
    assert bench.batch_launches(1, 4096, 4096, 74, True) == 75
    # spec-verify, 74 independent m = 16 calls: one run -> image + 3 grids
    assert scratch(16, 4096, 4096, 74, 2) == 256 * 4096 * 2
    assert bench.batch_launches(16, 4096, 4096, 74, True) == 1 + 3
    # the same calls dependent: no run, one small-m launch each
    assert scratch(16, 4096, 4096, 74, 0) == 0
    assert bench.batch_launches(16, 4096, 4096, 74, False) == 74
    # prefill (m = 512): no batch scratch; the first call's prepass, then GEMMs
    assert scratch(512, 7168, 7168, 4, 2) == 0
    assert bench.batch_launches(512, 7168, 7168, 4, True) == 5
    assert bench.batch_launches(512, 7168, 7168, 4, False) == 8


def test_x_planes_scratch_is_not_needed(lib):
    # the batched and routed GEMV launches convert x per thread: no scratch
    for k in (256, 4096, 16384, 16640):
        assert lib.q2k_x_planes_bytes(k, 3) == 0
    # a scratch argument is accepted and ignored: the call gets past every
    # argument check (it then fails only for want of a device here)
    x, w, y = 0x10000, 0x100000, 0x1000000
    args = (x, 3 * 256, w, 3 * 8 * 84, y, 3 * 8, 3, 1, 8, 256)
    st = lib.q2k_matmul_batched_mv(*args, 0x2000008, 16, None)
    assert st != INVALID, lib.q2k_last_error().decode()


def test_python_matmul_id_workspace_bytes_matches_the_library(lib):
    """The binding's workspace query is the library's (geometry only, no device)."""
    for n_tokens, top_k, n, k, experts in [(512, 8, 2048, 7168, 64), (33, 6, 8, 256, 8),
                                           (40, 2, 136, 1024, 4096)]:
        p = q2k.MatmulIdParams(n_tokens, top_k, n, k, experts, 10, n * (k // 256) * 84)
        for path in ("auto", "gemv", "tensor"):
            for slotted in (False, True):
                code = {"auto": q2k.PATH_AUTO, "gemv": q2k.PATH_GEMV, "tensor": q2k.PATH_TENSOR}[path]
                want = lib.q2k_matmul_id_workspace_bytes(code, q2k.ID_SLOTTED if slotted else 0,
                                                         ctypes.byref(p))
                got = q2k.matmul_id_workspace_bytes(n_tokens, top_k, n, k, experts, path=path,
                                                    slotted=slotted)
                assert got == want
