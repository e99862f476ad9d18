"""Python face of the CPU oracle in ``q2k_oracle.c`` (ctypes, numpy in/out).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check of the entry module and
the CPU-baseline leg of the benchmark may use this package; the product path
(the ``ggml_q2_quantized_gb300`` package and its CUDA library) never does.

What each call follows (mlx-native test page "tests/deepseek_q2_k.rs"):

* ``f16_to_f32``      - the binary16 decode of ``d``/``dmin`` (``half::f16::to_f32``).
* ``dequant_block``   - fn ``reference_dequant``: the canonical GGML loop order.
* ``dequantize``      - fn ``test_only_dequantize`` as the tests
                        ``q2_k_host_decode_*`` pin it (exact sizes or error).
* ``gather``          - test ``q2_k_embedding_gather_matches_canonical_rows_and_
                        rejects_bad_ids`` (rows by id; id >= vocab is an error).
* ``matmul``          - fn ``run_dense``'s expected value, ``y[m,n] = sum_k
                        x[m,k] w[n,k]``, summed in f64 instead of f32.
* ``matmul_batched_mv`` - test ``q2_k_batched_mv_is_byte_identical_to_
                        independent_dispatches``: batch b's matrix (at b n K/256
                        84 bytes) times batch b's input row, one ``matmul`` each.
* ``matmul_id``       - fn ``run_expert``'s expected value: route r = t top_k +
                        slot (token-major ids) takes token t's input and the
                        weights of expert ids[r] (at ids[r] expert_stride bytes);
                        an id >= n_experts is an error.  ``slotted``: route r
                        takes input row r instead (test ``q2_k_slotted_down_mm_
                        is_byte_identical_to_flattened_rows``: x [tokens, top_k,
                        k], the same values as the flattened call with top_k 1).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q2k_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libq2k_oracle.so")
_lock = threading.Lock()
_lib = None

QK_K = 256
BLOCK_BYTES = 84


class OracleError(ValueError):
    """A malformed input the oracle rejects (the pages' InvalidArgument)."""


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle source with gcc (no FMA contraction); return the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """One loaded build of the oracle library (the default one, or a variant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.q2ko_f16_to_f32.restype = ctypes.c_float
        lib.q2ko_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.q2ko_dequant_block.restype = None
        lib.q2ko_dequant_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.q2ko_dequantize.restype = ctypes.c_int
        lib.q2ko_dequantize.argtypes = [ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p, ctypes.c_size_t]
        lib.q2ko_gather.restype = ctypes.c_int
        lib.q2ko_gather.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32,
                                    ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]
        lib.q2ko_matmul.restype = ctypes.c_int
        lib.q2ko_matmul.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t,
                                    ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        self.lib = lib
        self.path = lib_path

    def f16_to_f32(self, bits) -> np.ndarray:
        """Decode uint16 binary16 bit patterns to float32, one call per value."""
        f = self.lib.q2ko_f16_to_f32
        bits = np.asarray(bits, dtype=np.uint16).reshape(-1)
        return np.array([f(int(b)) for b in bits], dtype=np.float32)

    def dequant_block(self, block: np.ndarray) -> np.ndarray:
        block = np.ascontiguousarray(block, dtype=np.uint8)
        if block.size != BLOCK_BYTES:
            raise OracleError(f"a Q2_K block is {BLOCK_BYTES} bytes, got {block.size}")
        out = np.empty(QK_K, dtype=np.float32)
        self.lib.q2ko_dequant_block(_ptr(block), _ptr(out))
        return out

    def dequantize(self, blocks: np.ndarray, n_out: int | None = None) -> np.ndarray:
        """Decode whole blocks; ``n_out`` (default: the exact count) must match."""
        blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
        if n_out is None:
            n_out = (blocks.size // BLOCK_BYTES) * QK_K
        out = np.empty(max(n_out, 1), dtype=np.float32)
        rc = self.lib.q2ko_dequantize(_ptr(blocks), blocks.size, _ptr(out), n_out)
        if rc != 0:
            raise OracleError("malformed Q2_K buffer")
        return out[:n_out]

    def gather(self, table: np.ndarray, vocab: int, embed_dim: int, ids) -> np.ndarray:
        table = np.ascontiguousarray(table, dtype=np.uint8).reshape(-1)
        ids = np.ascontiguousarray(ids, dtype=np.uint32).reshape(-1)
        if embed_dim % QK_K != 0:
            raise OracleError("embed_dim must be a multiple of 256")
        if table.size != vocab * (embed_dim // QK_K) * BLOCK_BYTES:
            raise OracleError("table size does not match vocab x embed_dim")
        out = np.empty((max(ids.size, 1), embed_dim), dtype=np.float32)
        rc = self.lib.q2ko_gather(_ptr(table), vocab, embed_dim, _ptr(ids), ids.size,
                                  _ptr(out))
        if rc == 2:
            raise OracleError("embedding id out of range")
        if rc != 0:
            raise OracleError("embed_dim must be a multiple of 256")
        return out[: ids.size]

    def matmul(self, x: np.ndarray, w: np.ndarray, n: int, threads: int = 1):
        """Return ``(y, s_abs)``, both float64 ``[M, n]``.

        ``y[m, r] = sum_k x[m, k] * w[r, k]`` with every weight decoded by the
        page's loop and the sum taken sequentially in f64; ``s_abs[m, r] =
        sum_k |x[m, k] * w[r, k]|``.
        """
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 2:
            raise OracleError("x must be [M, K]")
        M, K = x.shape
        w = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
        if K % QK_K != 0 or w.size != n * (K // QK_K) * BLOCK_BYTES:
            raise OracleError("K must be a multiple of 256 and w must hold n rows of "
                              "K/256 blocks")
        y = np.empty((M, n), dtype=np.float64)
        s_abs = np.empty((M, n), dtype=np.float64)
        threads = max(1, min(int(threads), 256, max(n, 1)))
        scratch = np.empty(threads * K, dtype=np.float32)
        rc = self.lib.q2ko_matmul(_ptr(x), _ptr(w), _ptr(y), _ptr(s_abs), M, n, K,
                                  threads, _ptr(scratch))
        if rc != 0:
            raise OracleError("oracle matmul failed")
        return y, s_abs


    # ---- batched and routed products: compositions of ``matmul`` ----------

    def matmul_batched_mv(self, x: np.ndarray, w: np.ndarray, n: int, threads: int = 1):
        """Return ``(y, s_abs)``, float64 ``[batches, n]``: row b is batch b's
        matrix (the b-th run of ``n * K/256`` blocks of ``w``) times ``x[b]``."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 2:
            raise OracleError("x must be [batches, K]")
        batches, K = x.shape
        wb = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
        per = n * (K // QK_K) * BLOCK_BYTES
        if K % QK_K != 0 or wb.size != batches * per:
            raise OracleError("w must hold one n x K matrix per batch")
        y = np.empty((batches, n), dtype=np.float64)
        s_abs = np.empty((batches, n), dtype=np.float64)
        for b in range(batches):
            yb, sb = self.matmul(x[b:b + 1], wb[b * per:(b + 1) * per], n, threads)
            y[b], s_abs[b] = yb[0], sb[0]
        return y, s_abs

    def route_token(self, route: int, top_k: int) -> int:
        """Token of route ``route``: the ids are token-major (t top_k + slot)."""
        return route // top_k

    def expert_bytes(self, w: np.ndarray, expert: int, n: int, K: int,
                     expert_stride: int) -> np.ndarray:
        """Expert ``expert``'s n x K matrix: ``n K/256`` blocks from byte
        ``expert * expert_stride``."""
        size = n * (K // QK_K) * BLOCK_BYTES
        start = expert * expert_stride
        if start + size > w.size:
            raise OracleError("expert matrix runs past the end of w")
        return w[start:start + size]

    def matmul_id(self, x: np.ndarray, w: np.ndarray, ids, n: int, n_experts: int,
                  expert_stride: int, top_k: int, threads: int = 1, slotted: bool = False):
        """Return ``(y, s_abs)``, float64 ``[n_tokens * top_k, n]``: row r is
        expert ``ids[r]``'s matrix times the input of token ``r // top_k`` (of
        route r itself when ``slotted``: x is then ``[n_tokens * top_k, K]``)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 2:
            raise OracleError("x must be [rows, K]")
        rows, K = x.shape
        ids = np.ascontiguousarray(ids, dtype=np.uint32).reshape(-1)
        n_tokens = rows // top_k if slotted and top_k >= 1 else rows
        if top_k < 1 or ids.size != n_tokens * top_k or K % QK_K != 0 or \
                (slotted and rows != ids.size):
            raise OracleError("ids must hold top_k experts per token and K a multiple of 256")
        wb = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1)
        y = np.empty((ids.size, n), dtype=np.float64)
        s_abs = np.empty((ids.size, n), dtype=np.float64)
        for r, e in enumerate(ids.tolist()):
            if e >= n_experts:
                raise OracleError(f"expert id {e} out of range (n_experts = {n_experts})")
            t = r if slotted else self.route_token(r, top_k)
            yr, sr = self.matmul(x[t:t + 1], self.expert_bytes(wb, e, n, K, expert_stride), n,
                                 threads)
            y[r], s_abs[r] = yr[0], sr[0]
        return y, s_abs


def default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def f16_to_f32(bits) -> np.ndarray:
    return default().f16_to_f32(bits)


def dequant_block(block: np.ndarray) -> np.ndarray:
    return default().dequant_block(block)


def dequantize(blocks: np.ndarray, n_out: int | None = None) -> np.ndarray:
    return default().dequantize(blocks, n_out)


def gather(table: np.ndarray, vocab: int, embed_dim: int, ids) -> np.ndarray:
    return default().gather(table, vocab, embed_dim, ids)


def matmul(x: np.ndarray, w: np.ndarray, n: int, threads: int = 1):
    return default().matmul(x, w, n, threads)


def matmul_rows(x: np.ndarray, w: np.ndarray, n: int, rows, threads: int = 1):
    """``matmul`` restricted to the weight rows ``rows`` (for sampled checks)."""
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    K = x.shape[1]
    row_bytes = (K // QK_K) * BLOCK_BYTES
    w2 = np.ascontiguousarray(w, dtype=np.uint8).reshape(n, row_bytes)[rows]
    return default().matmul(x, w2, rows.size, threads=threads)


def matmul_batched_mv(x: np.ndarray, w: np.ndarray, n: int, threads: int = 1):
    return default().matmul_batched_mv(x, w, n, threads)


def matmul_id(x: np.ndarray, w: np.ndarray, ids, n: int, n_experts: int, expert_stride: int,
              top_k: int, threads: int = 1, slotted: bool = False):
    return default().matmul_id(x, w, ids, n, n_experts, expert_stride, top_k, threads, slotted)
