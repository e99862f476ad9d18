"""GGML Q2_K weight-quantized matmul, dequantize and embedding gather on GB300.

A thin ctypes binding over the C ABI of ``libq2k.so`` (declared in
``include/q2k.h``).  It only marshals arguments: every step of the work runs in
the library's CUDA kernels on the tensors' device, on PyTorch's current stream.
PyTorch supplies device memory and streams, nothing else.  There is no CPU
fallback: if the library has not been built (``ggml_q2_quantized_gb300.build``)
or no sm_103 device is present, the calls raise.

Names follow the mlx-native page "tests/deepseek_q2_k.rs": ``matmul`` is
``quantized_matmul_ggml`` (with ``path=`` playing the role of
``dispatch_mm_for_test``), ``embedding_gather`` is ``embedding_gather_q2_k`` and
``dequantize`` is ``test_only_dequantize``.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

QK_K = 256
BLOCK_BYTES = 84
GGML_TYPE_Q2_K = 10

PATH_AUTO, PATH_GEMV, PATH_TENSOR = 0, 1, 2
FLAG_CONST_WEIGHTS = 1
FLAG_INDEPENDENT = 2
ID_SLOTTED = 1
_PATHS = {"auto": PATH_AUTO, "gemv": PATH_GEMV, "tensor": PATH_TENSOR,
          PATH_AUTO: PATH_AUTO, PATH_GEMV: PATH_GEMV, PATH_TENSOR: PATH_TENSOR}

STATUS = {0: "Q2K_OK", 1: "Q2K_ERR_INVALID_ARGUMENT", 2: "Q2K_ERR_BAD_ID",
          3: "Q2K_ERR_CUDA", 4: "Q2K_ERR_TIMEOUT", 5: "Q2K_ERR_NO_DEVICE", 6: "Q2K_ERR_IO"}

HEADER = os.path.join(_build.INCLUDE, "q2k.h")
LIB_PATH = _build.LIB_PATH


class Q2KError(RuntimeError):
    """A non-OK status from libq2k, with its message."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class InvalidArgument(Q2KError, ValueError):
    pass


class MatmulParams(ctypes.Structure):
    _fields_ = [("m", ctypes.c_uint32), ("n", ctypes.c_uint32), ("k", ctypes.c_uint32),
                ("ggml_type", ctypes.c_uint32)]


class MatmulIdParams(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_uint32), ("top_k", ctypes.c_uint32), ("n", ctypes.c_uint32),
                ("k", ctypes.c_uint32), ("n_experts", ctypes.c_uint32),
                ("ggml_type", ctypes.c_uint32), ("expert_stride", ctypes.c_uint64)]


class GgufTensor(ctypes.Structure):
    _fields_ = [("ggml_type", ctypes.c_uint32), ("n_dims", ctypes.c_uint32),
                ("dims", ctypes.c_uint64 * 4), ("n_elements", ctypes.c_uint64),
                ("offset", ctypes.c_uint64), ("byte_len", ctypes.c_uint64)]


class MatmulCall(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_elems", ctypes.c_size_t), ("w", ctypes.c_void_p),
                ("w_bytes", ctypes.c_size_t), ("y", ctypes.c_void_p), ("y_elems", ctypes.c_size_t),
                ("params", MatmulParams), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("path", ctypes.c_uint32),
                ("flags", ctypes.c_uint32)]


class EmbeddingParams(ctypes.Structure):
    _fields_ = [("vocab_size", ctypes.c_uint32), ("embed_dim", ctypes.c_uint32),
                ("n_tokens", ctypes.c_uint32), ("ggml_type", ctypes.c_uint32)]


_lock = threading.Lock()
_lib = None


def header_functions() -> list[str]:
    """Names of the functions ``include/q2k.h`` declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(q2k_\w+)\s*\(", text, flags=re.M)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the in-tree libq2k.so (built by ``build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libq2k is not built ({p} missing): run ggml_q2_quantized_gb300.build.build() "
                "- there is no fallback implementation")
        lib = ctypes.CDLL(p)
        vp, sz, u32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
        lib.q2k_dequantize.argtypes = [vp, sz, vp, sz, vp]
        lib.q2k_embedding_gather.argtypes = [vp, sz, vp, vp, sz, ctypes.POINTER(EmbeddingParams),
                                             vp, vp]
        lib.q2k_matmul.argtypes = [vp, sz, vp, sz, vp, sz, ctypes.POINTER(MatmulParams), vp]
        lib.q2k_matmul_path.argtypes = [ctypes.c_int, vp, sz, vp, sz, vp, sz,
                                        ctypes.POINTER(MatmulParams), vp]
        lib.q2k_matmul_ex.argtypes = [ctypes.c_int, ctypes.c_uint32, vp, sz, vp, sz, vp, sz,
                                      ctypes.POINTER(MatmulParams), vp, sz, vp]
        lib.q2k_matmul_workspace_bytes.argtypes = [ctypes.POINTER(MatmulParams), ctypes.c_int]
        lib.q2k_matmul_workspace_bytes.restype = ctypes.c_size_t
        lib.q2k_matmul_batched_mv.argtypes = [vp, sz, vp, sz, vp, sz, ctypes.c_uint32,
                                              ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                              vp, sz, vp]
        lib.q2k_matmul_id.argtypes = [vp, sz, vp, sz, vp, vp, sz, ctypes.POINTER(MatmulIdParams),
                                      vp, vp, sz, vp]
        lib.q2k_matmul_id_slotted.argtypes = lib.q2k_matmul_id.argtypes
        lib.q2k_matmul_id_pair.argtypes = [vp, sz, vp, sz, vp, sz, vp, vp, vp, sz,
                                           ctypes.POINTER(MatmulIdParams), vp, vp, sz, vp]
        lib.q2k_matmul_id_ex.argtypes = [ctypes.c_int, ctypes.c_uint32, vp, sz, vp, sz, vp, vp, sz,
                                         ctypes.POINTER(MatmulIdParams), vp, vp, sz, vp]
        lib.q2k_matmul_id_pair_ex.argtypes = [ctypes.c_int, vp, sz, vp, sz, vp, sz, vp, vp, vp, sz,
                                              ctypes.POINTER(MatmulIdParams), vp, vp, sz, vp]
        lib.q2k_matmul_id_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_uint32,
                                                      ctypes.POINTER(MatmulIdParams)]
        lib.q2k_matmul_id_workspace_bytes.restype = sz
        lib.q2k_x_planes_bytes.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
        lib.q2k_x_planes_bytes.restype = sz
        lib.q2k_gguf_open.argtypes = [ctypes.c_char_p, ctypes.POINTER(vp)]
        lib.q2k_gguf_close.argtypes = [vp]
        lib.q2k_gguf_close.restype = None
        lib.q2k_gguf_tensor_count.argtypes = [vp]
        lib.q2k_gguf_tensor_count.restype = ctypes.c_uint64
        lib.q2k_gguf_tensor_name.argtypes = [vp, ctypes.c_uint64]
        lib.q2k_gguf_tensor_name.restype = ctypes.c_char_p
        lib.q2k_gguf_tensor_info.argtypes = [vp, ctypes.c_char_p, ctypes.POINTER(GgufTensor)]
        lib.q2k_gguf_read_tensor.argtypes = [vp, ctypes.c_char_p, vp, sz]
        lib.q2k_matmul_ex_batch.argtypes = [ctypes.POINTER(MatmulCall), sz, vp, sz, vp]
        lib.q2k_matmul_batch_scratch_bytes.argtypes = [ctypes.POINTER(MatmulCall), sz]
        lib.q2k_matmul_batch_scratch_bytes.restype = sz
        lib.q2k_device_error.argtypes = [u32p, vp]
        lib.q2k_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        for fn in ("q2k_dequantize", "q2k_embedding_gather", "q2k_matmul", "q2k_matmul_path",
                   "q2k_matmul_ex", "q2k_matmul_ex_batch", "q2k_matmul_batched_mv", "q2k_matmul_id",
                   "q2k_matmul_id_slotted", "q2k_matmul_id_pair", "q2k_matmul_id_ex",
                   "q2k_matmul_id_pair_ex", "q2k_device_error",
                   "q2k_selftest_wait_timeout", "q2k_gguf_open", "q2k_gguf_tensor_info",
                   "q2k_gguf_read_tensor"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.q2k_last_error.restype = ctypes.c_char_p
        lib.q2k_last_error.argtypes = []
        lib.q2k_abi_version.restype = ctypes.c_int
        lib.q2k_abi_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def _check(lib, status: int):
    if status != 0:
        msg = lib.q2k_last_error().decode(errors="replace")
        if status == 1:
            raise InvalidArgument(status, msg)
        raise Q2KError(status, msg)


_torch_mod = None
_raw_stream = None


def _torch():
    global _torch_mod, _raw_stream
    if _torch_mod is None:
        import torch
        # the raw handle of a device's current stream without building a
        # torch.cuda.Stream object (the per-call cost of the public accessor)
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _torch_mod = torch
    return _torch_mod


def _stream_handle(tensor) -> int:
    torch = _torch()
    if _raw_stream is not None:
        return _raw_stream(tensor.device.index)
    return torch.cuda.current_stream(tensor.device).cuda_stream


class _on_device:
    """``torch.cuda.device(t.device)`` only when it is not already current."""

    __slots__ = ("idx", "prev")

    def __init__(self, tensor):
        self.idx = tensor.device.index
        self.prev = None

    def __enter__(self):
        torch = _torch()
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            _torch().cuda.set_device(self.prev)


def _require_cuda(t, name, dtype):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def dequantize(blocks, out=None):
    """Decode a uint8 CUDA tensor of whole Q2_K blocks to float32 (256 per block)."""
    torch = _torch()
    _require_cuda(blocks, "blocks", torch.uint8)
    n_out = (blocks.numel() // BLOCK_BYTES) * QK_K
    if out is None:
        out = torch.empty(max(n_out, 1), dtype=torch.float32, device=blocks.device)[:n_out]
    _require_cuda(out, "out", torch.float32)
    lib = load()
    with _on_device(blocks):
        _check(lib, lib.q2k_dequantize(blocks.data_ptr(), blocks.numel(), out.data_ptr(),
                                       out.numel(), _stream_handle(blocks)))
    return out


def embedding_gather(table, ids, embed_dim: int, vocab_size: int | None = None, out=None,
                     check: bool = True):
    """Rows ``ids`` of a Q2_K table ``[vocab, embed_dim]`` decoded to float32.

    With ``check`` (the default) the call waits for the stream and raises
    ``InvalidArgument`` if any id was >= vocab_size, as the pages' gather does;
    with ``check=False`` it returns ``(out, bad_id_count)`` without waiting.
    """
    torch = _torch()
    _require_cuda(table, "table", torch.uint8)
    _require_cuda(ids, "ids", ids.dtype)
    if ids.element_size() != 4 or ids.is_floating_point():
        raise TypeError("ids must be a 32-bit integer tensor (read as uint32)")
    row_bytes = (embed_dim // QK_K) * BLOCK_BYTES
    if vocab_size is None:
        vocab_size = table.numel() // row_bytes if row_bytes else 0
    n_tokens = ids.numel()
    if out is None:
        out = torch.empty((n_tokens, embed_dim), dtype=torch.float32, device=table.device)
    _require_cuda(out, "out", torch.float32)
    bad = torch.zeros(1, dtype=torch.int32, device=table.device)
    p = EmbeddingParams(vocab_size, embed_dim, n_tokens, GGML_TYPE_Q2_K)
    lib = load()
    with _on_device(table):
        _check(lib, lib.q2k_embedding_gather(table.data_ptr(), table.numel(), ids.data_ptr(),
                                             out.data_ptr(), out.numel(), ctypes.byref(p),
                                             bad.data_ptr(), _stream_handle(table)))
    if not check:
        return out, bad
    n_bad = int(bad.item())
    if n_bad:
        raise InvalidArgument(1, f"{n_bad} embedding id(s) >= vocab_size {vocab_size}")
    return out


_ws_bytes_cache: dict = {}


def matmul(x, w, n: int, out=None, path="auto", const_weights: bool = False,
           workspace="auto", independent: bool = False):
    """``y[m, r] = sum_k x[m, k] * W[r, k]`` with W = ``n`` rows of Q2_K blocks.

    ``const_weights=True`` passes Q2K_FLAG_CONST_WEIGHTS: the caller promises
    that the kernel enqueued just before on the stream does not write ``w``.
    ``independent=True`` passes Q2K_FLAG_INDEPENDENT: no kernel still running
    on the stream writes ``x`` or ``w`` or touches ``out`` (e.g. several
    projections of one activation enqueued back to back), so consecutive
    m = 1 calls overlap.
    ``workspace``: "auto" allocates the tensor-core path's workspace from
    PyTorch's caching allocator; None runs without one; or a uint8 CUDA tensor.
    """
    torch = _torch()
    _require_cuda(x, "x", torch.float32)
    _require_cuda(w, "w", torch.uint8)
    if x.dim() != 2:
        raise ValueError("x must be [m, k]")
    m, k = x.shape
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=x.device)
    _require_cuda(out, "out", torch.float32)
    p = MatmulParams(m, n, k, GGML_TYPE_Q2_K)
    lib = _lib if _lib is not None else load()
    pcode = _PATHS[path]
    ws_ptr, ws_bytes = None, 0
    if isinstance(workspace, str):
        # the GEMV path takes no workspace: skip the query for it
        if pcode == PATH_GEMV or (pcode == PATH_AUTO and m <= 8):
            workspace = None
        else:
            key = (m, n, k, pcode)
            need = _ws_bytes_cache.get(key)
            if need is None:
                need = lib.q2k_matmul_workspace_bytes(ctypes.byref(p), pcode)
                _ws_bytes_cache[key] = need
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device) if need else None
    if workspace is not None:
        _require_cuda(workspace, "workspace", torch.uint8)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    flags = (FLAG_CONST_WEIGHTS if const_weights else 0) | (FLAG_INDEPENDENT if independent else 0)
    with _on_device(x):
        _check(lib, lib.q2k_matmul_ex(pcode, flags, x.data_ptr(), x.numel(), w.data_ptr(),
                                      w.numel(), out.data_ptr(), out.numel(), ctypes.byref(p),
                                      ws_ptr, ws_bytes, _stream_handle(x)))
    return out


class MatmulBatch:
    """A fixed list of matmuls enqueued by one library call per ``run()``.

    ``calls`` holds dicts with the arguments of ``matmul``: ``x``, ``w``, ``n``
    and optionally ``out``, ``path``, ``const_weights``, ``independent``,
    ``workspace`` (a uint8 CUDA tensor; "auto" allocates one per distinct
    geometry, shared by its calls).  Everything is checked and packed once;
    ``run()`` enqueues all calls in order on the current stream of the first
    call's device with ``q2k_matmul_ex_batch`` (results bit-identical to
    separate ``matmul`` calls; m = 1 calls reading one x convert it once),
    except that independent tensor-path calls with m <= 64 on one x, enough
    of them to fill the GPU, share persistent grids over all of k (the tensor
    path's bound, deterministic, other bits than a separate call).  The
    tensors stay bound: update their contents in place between runs.  ``outs``
    lists the output tensors in call order.

    ``graph=True``: the first ``run()`` enqueues the calls and captures them
    into a CUDA graph; later runs replay it on the current stream, one launch
    from the host for the whole list (the same kernels and bits).
    """

    def __init__(self, calls, graph: bool = False):
        torch = _torch()
        calls = list(calls)
        self._lib = load()
        self._use_graph = bool(graph)
        self._graph = None
        self._arr = (MatmulCall * max(1, len(calls)))()
        self._keep = []
        self.outs = []
        shared_ws = {}
        for i, c in enumerate(calls):
            x, w, n = c["x"], c["w"], int(c["n"])
            _require_cuda(x, "x", torch.float32)
            _require_cuda(w, "w", torch.uint8)
            if x.dim() != 2:
                raise ValueError("x must be [m, k]")
            m, k = x.shape
            out = c.get("out")
            if out is None:
                out = torch.empty((m, n), dtype=torch.float32, device=x.device)
            _require_cuda(out, "out", torch.float32)
            pcode = _PATHS[c.get("path", "auto")]
            ws = c.get("workspace", "auto")
            p = MatmulParams(m, n, k, GGML_TYPE_Q2_K)
            if isinstance(ws, str):
                tensor_path = pcode == PATH_TENSOR or (pcode == PATH_AUTO and m > 8)
                ws = None
                if tensor_path:
                    need = self._lib.q2k_matmul_workspace_bytes(ctypes.byref(p), pcode)
                    if need:
                        key = (x.device.index, need)
                        if key not in shared_ws:
                            shared_ws[key] = torch.empty(need, dtype=torch.uint8, device=x.device)
                        ws = shared_ws[key]
            if ws is not None:
                _require_cuda(ws, "workspace", torch.uint8)
            flags = (FLAG_CONST_WEIGHTS if c.get("const_weights") else 0) | \
                    (FLAG_INDEPENDENT if c.get("independent") else 0)
            a = self._arr[i]
            a.x, a.x_elems, a.w, a.w_bytes = x.data_ptr(), x.numel(), w.data_ptr(), w.numel()
            a.y, a.y_elems, a.params = out.data_ptr(), out.numel(), p
            a.workspace = ws.data_ptr() if ws is not None else None
            a.workspace_bytes = ws.numel() if ws is not None else 0
            a.path, a.flags = pcode, flags
            self._keep.append((x, w, out, ws))
            self.outs.append(out)
        self._count = len(calls)
        # scratch for x converted once: the rows several m = 1 calls share, and
        # the bf16 image of each run of independent small-m tensor calls
        need = self._lib.q2k_matmul_batch_scratch_bytes(self._arr, self._count) if calls else 0
        self._scratch = (torch.empty(need, dtype=torch.uint8, device=calls[0]["x"].device)
                         if need else None)

    def _enqueue(self):
        with _on_device(self._keep[0][0]):
            sp = self._scratch
            _check(self._lib, self._lib.q2k_matmul_ex_batch(
                self._arr, self._count, sp.data_ptr() if sp is not None else None,
                sp.numel() if sp is not None else 0, _stream_handle(self._keep[0][0])))

    def run(self):
        if self._count == 0:
            return self.outs
        if not self._use_graph:
            self._enqueue()
            return self.outs
        if self._graph is not None:
            with _on_device(self._keep[0][0]):
                self._graph.replay()
            return self.outs
        torch = _torch()
        self._enqueue()  # this run; the graph serves the next ones
        dev = self._keep[0][0].device
        with _on_device(self._keep[0][0]):
            cur = torch.cuda.current_stream(dev)
            side = torch.cuda.Stream(dev)
            side.wait_stream(cur)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self._enqueue()
            cur.wait_stream(side)
        self._graph = g
        return self.outs


def _planes_scratch(lib, k, rows, device, scratch):
    """(pointer, bytes) of the x-planes scratch: "auto" allocates one."""
    if scratch is None:
        return None, 0, None
    if isinstance(scratch, str):
        need = lib.q2k_x_planes_bytes(k, rows)
        if not need:
            return None, 0, None
        scratch = _torch().empty(need, dtype=_torch().uint8, device=device)
    return scratch.data_ptr(), scratch.numel(), scratch


def matmul_batched_mv(x, w, n: int, out=None, scratch=None):
    """``batches`` matrix-vector products in one launch: ``x`` f32 ``[batches, k]``
    (or ``[batches, 1, k]``), ``w`` uint8 holding the batches' ``[n, k]`` Q2_K
    matrices back to back; returns ``[batches, n]`` (the shape of ``x`` with k
    replaced by n).  Each batch is bit-identical to ``matmul`` of it alone.
    ``scratch="auto"`` converts each batch's x once instead of per CTA (an
    extra launch; it pays for long k), or pass a uint8 tensor of
    ``q2k_x_planes_bytes(k, batches)`` bytes."""
    torch = _torch()
    _require_cuda(x, "x", torch.float32)
    _require_cuda(w, "w", torch.uint8)
    k = x.shape[-1]
    batches = x.shape[0]
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (n,), dtype=torch.float32, device=x.device)
    _require_cuda(out, "out", torch.float32)
    lib = load()
    sp, sb, _keep = _planes_scratch(lib, k, batches, x.device, scratch)
    with _on_device(x):
        _check(lib, lib.q2k_matmul_batched_mv(x.data_ptr(), x.numel(), w.data_ptr(), w.numel(),
                                              out.data_ptr(), out.numel(), batches, 1, n, k, sp, sb,
                                              _stream_handle(x)))
    return out


def _routed_finish(bad, check, outs, n_experts):
    if not check:
        return (*outs, bad) if len(outs) > 1 else (outs[0], bad)
    n_bad = int(bad.item())
    if n_bad:
        raise InvalidArgument(1, f"{n_bad} expert id(s) >= n_experts {n_experts}")
    return outs if len(outs) > 1 else outs[0]


def matmul_id_slotted(x, w, ids, n: int, n_experts: int, expert_stride: int | None = None,
                      out=None, check: bool = True, scratch=None):
    """Routed product with one input row per route: ``x`` f32 ``[n_tokens, top_k,
    k]``, ``ids`` ``[n_tokens, top_k]``; returns ``[n_tokens, top_k, n]``, route
    (t, s) = expert ``ids[t, s]`` times ``x[t, s]``.  ``check`` as ``matmul_id``."""
    torch = _torch()
    _require_cuda(x, "x", torch.float32)
    _require_cuda(w, "w", torch.uint8)
    _require_cuda(ids, "ids", ids.dtype)
    if ids.element_size() != 4 or ids.is_floating_point():
        raise TypeError("ids must be a 32-bit integer tensor (read as uint32)")
    n_tokens, top_k, k = x.shape
    if expert_stride is None:
        expert_stride = n * (k // QK_K) * BLOCK_BYTES
    if out is None:
        out = torch.empty((n_tokens, top_k, n), dtype=torch.float32, device=x.device)
    _require_cuda(out, "out", torch.float32)
    bad = torch.zeros(1, dtype=torch.int32, device=x.device)
    p = MatmulIdParams(n_tokens, top_k, n, k, n_experts, GGML_TYPE_Q2_K, expert_stride)
    lib = load()
    sp, sb, _keep = _planes_scratch(lib, k, n_tokens * top_k, x.device, scratch)
    with _on_device(x):
        _check(lib, lib.q2k_matmul_id_slotted(x.data_ptr(), x.numel(), w.data_ptr(), w.numel(),
                                              ids.data_ptr(), out.data_ptr(), out.numel(),
                                              ctypes.byref(p), bad.data_ptr(), sp, sb,
                                              _stream_handle(x)))
    return _routed_finish(bad, check, (out,), n_experts)


def matmul_id_pair(x, w_a, w_b, ids, n: int, n_experts: int, top_k: int,
                   expert_stride: int | None = None, check: bool = True, scratch="auto",
                   path=None, workspace=None):
    """Two routed products sharing ``x`` and ``ids`` (e.g. the gate and up
    projections) in one launch; returns ``(y_a, y_b)`` as ``matmul_id`` would.
    ``path`` ("gemv", "tensor" or "auto", as ``matmul_id_ex``) goes through
    ``q2k_matmul_id_pair_ex``; the tensor path routes and gathers x once for
    both products.  ``workspace`` as in ``matmul_id_ex``."""
    torch = _torch()
    _require_cuda(x, "x", torch.float32)
    _require_cuda(w_a, "w_a", torch.uint8)
    _require_cuda(w_b, "w_b", torch.uint8)
    _require_cuda(ids, "ids", ids.dtype)
    if ids.element_size() != 4 or ids.is_floating_point():
        raise TypeError("ids must be a 32-bit integer tensor (read as uint32)")
    n_tokens, k = x.shape
    if expert_stride is None:
        expert_stride = n * (k // QK_K) * BLOCK_BYTES
    y_a = torch.empty((ids.numel(), n), dtype=torch.float32, device=x.device)
    y_b = torch.empty((ids.numel(), n), dtype=torch.float32, device=x.device)
    bad = torch.zeros(1, dtype=torch.int32, device=x.device)
    p = MatmulIdParams(n_tokens, top_k, n, k, n_experts, GGML_TYPE_Q2_K, expert_stride)
    lib = load()
    if path is not None:
        pcode = _PATHS[path]
        if workspace is None:
            nbytes = lib.q2k_matmul_id_workspace_bytes(pcode, 0, ctypes.byref(p))
            if nbytes:
                workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
        wp = workspace.data_ptr() if workspace is not None else None
        wb = workspace.numel() if workspace is not None else 0
        with _on_device(x):
            _check(lib, lib.q2k_matmul_id_pair_ex(pcode, x.data_ptr(), x.numel(), w_a.data_ptr(),
                                                  w_a.numel(), w_b.data_ptr(), w_b.numel(),
                                                  ids.data_ptr(), y_a.data_ptr(), y_b.data_ptr(),
                                                  y_a.numel(), ctypes.byref(p), bad.data_ptr(),
                                                  wp, wb, _stream_handle(x)))
        return _routed_finish(bad, check, (y_a, y_b), n_experts)
    sp, sb, _keep = _planes_scratch(lib, k, n_tokens, x.device, scratch)
    with _on_device(x):
        _check(lib, lib.q2k_matmul_id_pair(x.data_ptr(), x.numel(), w_a.data_ptr(), w_a.numel(),
                                           w_b.data_ptr(), w_b.numel(), ids.data_ptr(),
                                           y_a.data_ptr(), y_b.data_ptr(), y_a.numel(),
                                           ctypes.byref(p), bad.data_ptr(), sp, sb,
                                           _stream_handle(x)))
    return _routed_finish(bad, check, (y_a, y_b), n_experts)


def matmul_id(x, w, ids, n: int, n_experts: int, top_k: int, expert_stride: int | None = None,
              out=None, check: bool = True, scratch="auto"):
    """Expert-routed product: ``x`` f32 ``[n_tokens, k]``, ``ids`` 32-bit ints
    ``[n_tokens * top_k]`` (token-major), expert e's ``[n, k]`` Q2_K matrix at
    byte ``e * expert_stride`` of ``w`` (default: packed, ``n * k/256 * 84``).
    Returns ``[n_tokens * top_k, n]`` with row r = expert ``ids[r]`` times token
    ``r // top_k``.  With ``check`` the call waits and raises ``InvalidArgument``
    if an id was >= n_experts; with ``check=False`` it returns ``(out,
    bad_id_count)`` without waiting."""
    torch = _torch()
    _require_cuda(x, "x", torch.float32)
    _require_cuda(w, "w", torch.uint8)
    _require_cuda(ids, "ids", ids.dtype)
    if ids.element_size() != 4 or ids.is_floating_point():
        raise TypeError("ids must be a 32-bit integer tensor (read as uint32)")
    n_tokens, k = x.shape
    if expert_stride is None:
        expert_stride = n * (k // QK_K) * BLOCK_BYTES
    if out is None:
        out = torch.empty((ids.numel(), n), dtype=torch.float32, device=x.device)
    _require_cuda(out, "out", torch.float32)
    bad = torch.zeros(1, dtype=torch.int32, device=x.device)
    p = MatmulIdParams(n_tokens, top_k, n, k, n_experts, GGML_TYPE_Q2_K, expert_stride)
    lib = load()
    sp, sb, _keep = _planes_scratch(lib, k, n_tokens, x.device, scratch)
    with _on_device(x):
        _check(lib, lib.q2k_matmul_id(x.data_ptr(), x.numel(), w.data_ptr(), w.numel(),
                                      ids.data_ptr(), out.data_ptr(), out.numel(),
                                      ctypes.byref(p), bad.data_ptr(), sp, sb, _stream_handle(x)))
    if not check:
        return out, bad
    n_bad = int(bad.item())
    if n_bad:
        raise InvalidArgument(1, f"{n_bad} expert id(s) >= n_experts {n_experts}")
    return out


def matmul_id_ex(x, w, ids, n: int, n_experts: int, top_k: int = 1, path="auto",
                 slotted: bool = False, expert_stride: int | None = None, out=None,
                 check: bool = True, workspace=None):
    """``matmul_id`` (or, with ``slotted``, ``matmul_id_slotted``; then ``x`` is
    ``[n_tokens, top_k, k]`` and ``top_k`` is taken from it) on a chosen path:
    ``"gemv"`` (fp32, as ``matmul_id``), ``"tensor"`` (routes grouped per
    expert and multiplied on the bf16 tensor cores) or ``"auto"`` (tensor above
    32 tokens).  ``workspace``: a CUDA uint8 tensor of at least
    ``matmul_id_workspace_bytes`` bytes, allocated here when None."""
    torch = _torch()
    _require_cuda(x, "x", torch.float32)
    _require_cuda(w, "w", torch.uint8)
    _require_cuda(ids, "ids", ids.dtype)
    if ids.element_size() != 4 or ids.is_floating_point():
        raise TypeError("ids must be a 32-bit integer tensor (read as uint32)")
    if slotted:
        n_tokens, top_k, k = x.shape
        shape = (n_tokens, top_k, n)
    else:
        n_tokens, k = x.shape
        shape = (n_tokens * top_k, n)
    if expert_stride is None:
        expert_stride = n * (k // QK_K) * BLOCK_BYTES
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=x.device)
    _require_cuda(out, "out", torch.float32)
    bad = torch.zeros(1, dtype=torch.int32, device=x.device)
    p = MatmulIdParams(n_tokens, top_k, n, k, n_experts, GGML_TYPE_Q2_K, expert_stride)
    pcode = _PATHS[path]
    flags = ID_SLOTTED if slotted else 0
    lib = load()
    if workspace is None:
        nbytes = lib.q2k_matmul_id_workspace_bytes(pcode, flags, ctypes.byref(p))
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    wp = workspace.data_ptr() if workspace is not None else None
    wb = workspace.numel() if workspace is not None else 0
    with _on_device(x):
        _check(lib, lib.q2k_matmul_id_ex(pcode, flags, x.data_ptr(), x.numel(), w.data_ptr(),
                                         w.numel(), ids.data_ptr(), out.data_ptr(), out.numel(),
                                         ctypes.byref(p), bad.data_ptr(), wp, wb,
                                         _stream_handle(x)))
    return _routed_finish(bad, check, (out,), n_experts)


def matmul_id_workspace_bytes(n_tokens: int, top_k: int, n: int, k: int, n_experts: int,
                              path="auto", slotted: bool = False,
                              expert_stride: int | None = None) -> int:
    """Bytes of workspace ``matmul_id_ex`` takes on ``path`` (0: none or invalid)."""
    if expert_stride is None:
        expert_stride = n * (k // QK_K) * BLOCK_BYTES
    p = MatmulIdParams(n_tokens, top_k, n, k, n_experts, GGML_TYPE_Q2_K, expert_stride)
    return int(load().q2k_matmul_id_workspace_bytes(_PATHS[path], ID_SLOTTED if slotted else 0,
                                                    ctypes.byref(p)))


class GgufFile:
    """An open GGUF file (host only): ``names``, ``info(name)`` (a ``GgufTensor``:
    ggml_type, n_dims, dims innermost first, n_elements, offset, byte_len),
    ``read(name)`` (the bytes as a numpy uint8 array) and ``to_device(name)``
    (those bytes in a CUDA uint8 tensor, ready for ``matmul`` when the type is
    Q2_K).  Use as a context manager or call ``close``."""

    def __init__(self, path):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib, self._lib.q2k_gguf_open(os.fsencode(path), ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h is not None and self._h.value:
            self._lib.q2k_gguf_close(self._h)
        self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def names(self) -> list[str]:
        n = self._lib.q2k_gguf_tensor_count(self._h)
        return [self._lib.q2k_gguf_tensor_name(self._h, i).decode() for i in range(n)]

    def info(self, name: str) -> GgufTensor:
        out = GgufTensor()
        _check(self._lib, self._lib.q2k_gguf_tensor_info(self._h, name.encode(), ctypes.byref(out)))
        return out

    def read(self, name: str):
        import numpy as np
        n = self.info(name).byte_len
        buf = np.empty(n, dtype=np.uint8)
        _check(self._lib, self._lib.q2k_gguf_read_tensor(self._h, name.encode(),
                                                         buf.ctypes.data, n))
        return buf

    def to_device(self, name: str, device="cuda"):
        torch = _torch()
        return torch.from_numpy(self.read(name)).to(device)


def selftest_wait_timeout(limit_us: int = 2000, device=None) -> None:
    """Enqueue the library's bounded-wait self-test on the current stream: a kernel
    waits ~limit_us on a barrier nothing completes, gives up and sets the time-out
    bit that ``device_error()`` then returns."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    lib = load()
    with torch.cuda.device(dev):
        _check(lib, lib.q2k_selftest_wait_timeout(int(limit_us),
                                                  torch.cuda.current_stream(dev).cuda_stream))


def device_error(device=None) -> int:
    """Read and clear the device error word (nonzero: a kernel gave up waiting)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    v = ctypes.c_uint32(0)
    lib = load()
    with torch.cuda.device(dev):
        _check(lib, lib.q2k_device_error(ctypes.byref(v),
                                         torch.cuda.current_stream(dev).cuda_stream))
    return int(v.value)
