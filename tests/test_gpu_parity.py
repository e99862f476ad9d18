"""GPU parity: every libq2k kernel against the CPU oracle on the same seeded inputs.

Tolerances (per output, S = sum_k |x[m,k] w[n,k]| from the oracle):
  dequantize / gather       bit-exact f32
  fp32 GEMV path            |y - y_ref| <= 1e-5 * S
  bf16 tensor-core path     |y - y_ref| <= 8e-3 * S
The bf16 bound is guaranteed for a correct kernel: rounding both operands to
bf16 costs at most (2u + u^2)|x w| per term with u = 2^-9 (3.92e-3), plus the
fp32 accumulation.
"""

import ctypes

import numpy as np
import pytest

import oracle
import q2k_workloads as wl

torch = pytest.importorskip("torch")
import ggml_q2_quantized_gb300 as q2k  # noqa: E402
from ggml_q2_quantized_gb300 import build as q2k_build  # noqa: E402

pytestmark = pytest.mark.gpu

TOL_GEMV = 1e-5
TOL_TC = 8e-3
ORACLE_THREADS = 16


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    q2k_build.build()
    q2k.load()
    yield
    assert q2k.device_error() == 0, "a kernel gave up waiting on a barrier"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_matmul(x, w, n, path):
    y = q2k.matmul(dev(x), dev(w), n, path=path)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def assert_close(y, yref, s, tol, what):
    err = np.abs(y - yref)
    bad = err > tol * s
    assert not np.isnan(y).any(), f"{what}: NaN in output"
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first {tuple(i)}: "
                             f"got {y[tuple(i)]}, want {yref[tuple(i)]}, S={s[tuple(i)]}")
    return float((err / np.maximum(s, 1e-300)).max())


def check_matmul(seed, m, n, k, path, tol):
    x, w = wl.make_matmul_inputs(seed, m, n, k)
    y = run_matmul(x, w, n, path)
    yref, s = oracle.matmul(x, w, n, threads=ORACLE_THREADS)
    return assert_close(y, yref, s, tol, f"{path} m={m} n={n} k={k}")


# ------------------------------------------------------------------ dequantize

def test_dequantize_page_block5_bit_exact():
    b = wl.page_block(5)
    out = q2k.dequantize(dev(b)).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), oracle.dequantize(b).view(np.uint32))


@pytest.mark.parametrize("n_blocks", [1, 8, 33, 10007])
def test_dequantize_random_bit_exact(n_blocks):
    rng = np.random.default_rng(n_blocks)
    blocks = wl.random_blocks(rng, n_blocks)
    out = q2k.dequantize(dev(blocks)).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), oracle.dequantize(blocks).view(np.uint32))


def test_dequantize_tiny_workload_bit_exact():
    inp = wl.make_inputs(wl.WORKLOADS[0])
    out = q2k.dequantize(dev(inp.w)).cpu().numpy()
    assert out.size == 8 * 256
    assert np.array_equal(out.view(np.uint32), oracle.dequantize(inp.w).view(np.uint32))


def test_dequantize_special_scales_bit_exact():
    # subnormal, max and zero d/dmin; every (sc, m) nibble pair
    rng = np.random.default_rng(3)
    blocks = wl.random_blocks(rng, 64).reshape(64, 84)
    for i, (d, dm) in enumerate([(0x0001, 0x03FF), (0x7BFF, 0x7BFF), (0, 0), (0x3C00, 0x0400)]):
        blocks[i, 80:82] = [d & 0xFF, d >> 8]
        blocks[i, 82:84] = [dm & 0xFF, dm >> 8]
    blocks[4:20, 0:16] = np.arange(256, dtype=np.uint8).reshape(16, 16)
    flat = blocks.reshape(-1)
    out = q2k.dequantize(dev(flat)).cpu().numpy()
    assert np.array_equal(out.view(np.uint32), oracle.dequantize(flat).view(np.uint32))


def _same_or_both_nan(a, b):
    """Bit-equal, except that any NaN matches any NaN (payloads are not specified)."""
    a, b = a.reshape(-1), b.reshape(-1)
    nan = np.isnan(a)
    return np.array_equal(nan, np.isnan(b)) and np.array_equal(a[~nan].view(np.uint32),
                                                               b[~nan].view(np.uint32))


# d or dmin = +Inf, -Inf or NaN (binary16 0x7C00, 0xFC00, 0x7E00), beside finite ones
NONFINITE_SCALES = [(0x7C00, 0x3C00), (0x3C00, 0x7C00), (0xFC00, 0x2E66), (0x2E66, 0xFC00),
                    (0x7E00, 0x3C00), (0x3C00, 0x7E00), (0x7C00, 0x7C00), (0x7C00, 0xFC00),
                    (0x0000, 0x7C00), (0x7C00, 0x0000), (0x7E00, 0x7E00)]


def _nonfinite_blocks(seed):
    rng = np.random.default_rng(seed)
    blocks = wl.random_blocks(rng, 2 * len(NONFINITE_SCALES)).reshape(-1, 84)
    for i, (d, dm) in enumerate(NONFINITE_SCALES):
        blocks[2 * i, 80:82] = [d & 0xFF, d >> 8]
        blocks[2 * i, 82:84] = [dm & 0xFF, dm >> 8]
    blocks[1::4, 0:16] = 0x00          # sc = m = 0 beside an infinite scale: inf * 0
    blocks[2::4, 16:80] = 0x00         # q = 0 everywhere
    return blocks


def test_dequantize_nonfinite_scales_match_oracle():
    """Blocks whose d or dmin is +-Inf or NaN decode as the page's f32 loop
    does (IEEE: inf * 0 = NaN, inf - inf = NaN); NaNs compared as NaN."""
    flat = _nonfinite_blocks(41).reshape(-1)
    out = q2k.dequantize(dev(flat)).cpu().numpy()
    want = oracle.dequantize(flat)
    assert np.isnan(want).any() and np.isinf(want).any()
    assert _same_or_both_nan(out, want)


def test_gather_nonfinite_scales_match_oracle():
    blocks = _nonfinite_blocks(42)
    vocab = blocks.shape[0] // 2   # rows of 512 (two blocks)
    table = blocks.reshape(-1)
    ids = np.array([0, vocab - 1, 3, 3, 1], dtype=np.uint32)
    out = q2k.embedding_gather(dev(table), dev(ids.astype(np.int32)), 512).cpu().numpy()
    want = oracle.gather(table, vocab, 512, ids)
    assert _same_or_both_nan(out, want)


def test_dequantize_rejects_malformed_on_device():
    b = dev(wl.page_block(1))
    with pytest.raises(q2k.InvalidArgument):
        q2k.dequantize(b[:83])
    out = torch.empty(255, dtype=torch.float32, device="cuda")
    with pytest.raises(q2k.InvalidArgument):
        q2k.dequantize(b, out=out)


def test_dequantize_guard_bands():
    rng = np.random.default_rng(9)
    blocks = wl.random_blocks(rng, 5)
    pad = 1024
    buf = torch.full((pad + 5 * 256 + pad,), float("nan"), device="cuda")
    q2k.dequantize(dev(blocks), out=buf[pad:pad + 5 * 256])
    host = buf.cpu().numpy()
    assert np.isnan(host[:pad]).all() and np.isnan(host[-pad:]).all()
    assert np.array_equal(host[pad:-pad].view(np.uint32), oracle.dequantize(blocks).view(np.uint32))


# ------------------------------------------------------------------ gather

def test_gather_page_case_and_bad_id():
    table = np.concatenate([wl.page_block(r + 2) for r in range(3)])
    t = dev(table)
    ids = dev(np.array([2, 0], dtype=np.int32))
    out = q2k.embedding_gather(t, ids, 256).cpu().numpy()
    want = oracle.gather(table, 3, 256, [2, 0])
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))
    with pytest.raises(q2k.InvalidArgument):
        q2k.embedding_gather(t, dev(np.array([2, 3], dtype=np.int32)), 256)
    out, bad = q2k.embedding_gather(t, dev(np.array([3, 1], dtype=np.int32)), 256, check=False)
    torch.cuda.synchronize()
    assert int(bad.item()) == 1
    host = out.cpu().numpy()
    assert (host[0] == 0).all()
    assert np.array_equal(host[1], oracle.dequant_block(wl.page_block(3)))


def test_gather_tiny_workload():
    inp = wl.make_inputs(wl.WORKLOADS[0])
    out = q2k.embedding_gather(dev(inp.table), dev(inp.ids.astype(np.int32)), 256).cpu().numpy()
    want = oracle.gather(inp.table, 8, 256, inp.ids)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))


def test_gather_spec_verify_workload():
    w = wl.WORKLOADS[3]
    inp = wl.make_inputs(w)
    out = q2k.embedding_gather(dev(inp.table), dev(inp.ids.astype(np.int32)), w.k).cpu().numpy()
    want = oracle.gather(inp.table, w.gather_vocab, w.k, inp.ids)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))


def test_gather_repeated_and_last_ids():
    rng = np.random.default_rng(4)
    vocab, dim = 37, 768
    table = wl.random_blocks(rng, vocab * 3)
    ids = np.array([36, 36, 0, 5, 36, 1], dtype=np.uint32)
    out = q2k.embedding_gather(dev(table), dev(ids.astype(np.int32)), dim).cpu().numpy()
    want = oracle.gather(table, vocab, dim, ids)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------------------ GEMV path

@pytest.mark.parametrize("m,n,k", [
    (1, 8, 256), (1, 1, 256), (1, 7, 512), (1, 9, 768), (1, 1000, 1280), (1, 333, 4096),
    (2, 100, 1024), (3, 65, 2304), (4, 8, 256), (5, 257, 512), (7, 31, 3072), (8, 129, 4096),
    (9, 40, 512), (17, 24, 1024),
])
def test_gemv_parity(m, n, k):
    check_matmul(1000 + m * 7 + n + k, m, n, k, "gemv", TOL_GEMV)


def test_gemv_page_run_dense_rows1():
    """Page fn run_dense(1): n = 8 rows block(r+1), x = input(1); the page's 2e-4."""
    w = np.concatenate([wl.page_block(r + 1) for r in range(8)])
    x = wl.page_input(1)
    y = run_matmul(x, w, 8, "auto")
    yref, s = oracle.matmul(x, w, 8)
    assert np.abs(y - yref).max() <= 2e-4
    assert_close(y, yref, s, TOL_GEMV, "run_dense(1)")


@pytest.mark.parametrize("name", ["tiny", "decode_gemv_4096", "ffn_pair", "ffn_pair_down"])
def test_gemv_workloads_full(name):
    w = wl.by_name(name)
    inp = wl.make_inputs(w, with_gather=False)
    y = run_matmul(inp.x, inp.w, w.n, "auto")
    yref, s = oracle.matmul(inp.x, inp.w, w.n, threads=ORACLE_THREADS)
    ratio = assert_close(y, yref, s, TOL_GEMV, name)
    print(f"{name}: max |y - y_ref| / S = {ratio:.3e}")


# ------------------------------------------------------------------ tensor-core path

@pytest.mark.parametrize("m,n,k", [
    (9, 8, 256),        # the page's forced-mm shape
    (1, 8, 256), (4, 64, 512), (16, 64, 256), (16, 100, 768),
    (127, 65, 512), (128, 128, 1024), (129, 200, 256), (300, 1000, 512),
    (16, 12288, 256),   # dispatcher picks 128-row weight tiles
    (130, 10000, 256),  # 192-row weight tiles, ragged last tile
    (200, 300, 512),    # ragged x tile (72 rows) and weight tile
    (257, 520, 1024),   # 1-row last x tile, 256-row weight tiles with a ragged one
    (384, 2000, 768),   # several waves of 128-row weight tiles
    (300, 20000, 1024), # 256-row x tiles (one ragged: 48 rows), TMA weight boxes, ragged N
])
def test_tensor_parity(m, n, k):
    check_matmul(2000 + m + n + k, m, n, k, "tensor", TOL_TC)


@pytest.mark.parametrize("m,n,k", [
    (1, 4096, 4096),    # 16-row x tile, 4 K parts (cluster of 4)
    (8, 8, 256),        # one part, no cluster
    (17, 333, 2560),    # 32-row x tile, 8 uneven parts of 1 or 2 blocks, ragged N
    (48, 129, 768),     # 64-row x tile (48 used), 3 parts
    (64, 4096, 4096),   # full 64-row x tile, 4 parts
    (16, 14336, 4096),  # one part, 112 CTAs, all 64 K stages of x resident
])
def test_tensor_small_m_parity(m, n, k):
    """m <= 64: x converted to bf16 in the GEMM, K parts summed in the cluster."""
    check_matmul(2500 + m + n + k, m, n, k, "tensor", TOL_TC)


@pytest.mark.parametrize("m,n,k", [
    (64, 4000, 8192),   # x capacity forces 7 parts (a cluster of 7) where 4 were asked
    (32, 14336, 4096),  # 2 parts where 1 was asked: 224 CTAs, more than one wave
    (33, 300, 14336),   # x does not fit even in 8 parts: the x-image path
])
def test_tensor_small_m_sampled_rows(m, n, k):
    x, w = wl.make_matmul_inputs(2600 + m, m, n, k)
    y = run_matmul(x, w, n, "tensor")
    rng = np.random.default_rng(m)
    rows = np.unique(np.concatenate([rng.choice(n, 48, replace=False), [0, 127, 128, n - 1]]))
    yref, s = oracle.matmul_rows(x, w, n, rows, threads=ORACLE_THREADS)
    assert_close(y[:, rows], yref, s, TOL_TC, f"m={m} n={n} k={k} sampled")


def test_matmul_batch_shared_image_independent_calls():
    """Consecutive independent tensor calls on one x (same m, k, workspace) in a
    batch: the later ones reuse the x image the first one converted and may run
    beside each other.  Each output is bit-identical to its own call and within
    the tensor path's bound of the oracle; 256- and 128-row x tiles, a ragged
    last weight tile, and a call on another x in between (which converts anew)."""
    for m, k, ns in ((512, 1024, (1024, 640, 1000, 1024)), (200, 768, (4096, 333, 4096))):
        x, _ = wl.make_matmul_inputs(3400 + m, m, 16, k)
        xd = dev(x)
        ws_list, calls, ref, refs_np = [], [], [], []
        for i, n in enumerate(ns):
            _, w = wl.make_matmul_inputs(3500 + m + i, m, n, k)
            wd = dev(w)
            calls.append(dict(x=xd, w=wd, n=n, path="tensor", independent=True))
            ref.append(q2k.matmul(xd, wd, n, path="tensor", independent=True))
            refs_np.append((w, n))
        # a call on another x between two calls on xd: the one after it converts again
        x2, w2 = wl.make_matmul_inputs(3600 + m, m, 256, k)
        calls.insert(2, dict(x=dev(x2), w=dev(w2), n=256, path="tensor", independent=True))
        ref.insert(2, q2k.matmul(dev(x2), dev(w2), 256, path="tensor", independent=True))
        torch.cuda.synchronize()
        for run in range(2):
            outs = q2k.MatmulBatch(calls).run()
            torch.cuda.synchronize()
            for i, (a, b) in enumerate(zip(outs, ref)):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"m={m} call {i} run {run}"
        rows = np.arange(0, 16)
        for (w, n), y in zip(refs_np, [o for j, o in enumerate(outs) if j != 2]):
            yref, s_ = oracle.matmul_rows(x, w, n, rows[rows < n], threads=ORACLE_THREADS)
            assert_close(y.cpu().numpy()[:, rows[rows < n]], yref, s_, TOL_TC, f"m={m} n={n} sampled")


def test_matmul_batch_small_m_runs_persistent():
    """Independent small-m tensor calls on one x in a batch, enough tiles to
    fill the GPU: the run shares persistent grids over all of k (x converted
    once into the batch scratch).  Every output within the tensor path's bound
    of the oracle on sampled weight rows (tile edges and the ragged last tile
    included), and bit-identical on a second run.  Cases: x resident in shared
    memory (m = 16, k = 4096) with a ragged call; the x ring (m = 40, k = 2048,
    and m = 16, k = 14336); m = 5 forced onto the tensor path; more than 32
    calls (two grids, the second on the ready image); a call on another x in
    the middle splits the run."""
    cases = [
        (16, 4096, [4096] * 4 + [1000], {}),
        (40, 2048, [4096] * 4 + [333], {}),
        (16, 14336, [4096] * 4, {}),
        (5, 1024, [2048] * 10, dict(path="tensor")),
        (24, 1024, [512] * 36 + [200], {}),
    ]
    for ci, (m, k, ns, kw) in enumerate(cases):
        x, _ = wl.make_matmul_inputs(4100 + ci, m, 16, k)
        xd = dev(x)
        calls, ws_np = [], []
        for i, n in enumerate(ns):
            _, w = wl.make_matmul_inputs(4200 + 50 * ci + i, m, n, k)
            calls.append(dict(x=xd, w=dev(w), n=n, independent=True, **kw))
            ws_np.append((w, n))
        batch = q2k.MatmulBatch(calls)
        assert batch._scratch is not None, f"case {ci}: no run formed"
        outs = [o.clone() for o in batch.run()]
        torch.cuda.synchronize()
        for o in batch.outs:
            o.fill_(float("nan"))
        again = batch.run()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(again, outs)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"case {ci} call {i} rerun"
        rng = np.random.default_rng(4300 + ci)
        for i, ((w, n), y) in enumerate(zip(ws_np, outs)):
            if len(ns) > 8 and i % 7 and i != len(ns) - 1:
                continue   # a sample of the many calls
            pick = rng.choice(n, min(n, 24), replace=False)
            rows = np.unique(np.concatenate([pick, [0, min(127, n - 1), min(128, n - 1), n - 1]]))
            yref, s_ = oracle.matmul_rows(x, w, n, rows, threads=ORACLE_THREADS)
            assert_close(y.cpu().numpy()[:, rows], yref, s_, TOL_TC, f"case {ci} (m={m} k={k}) call {i}")
    # a call on another x splits the run: both parts still correct
    m, k = 16, 1024
    x, _ = wl.make_matmul_inputs(4400, m, 16, k)
    x2, w2 = wl.make_matmul_inputs(4401, m, 256, k)
    xd = dev(x)
    calls, ws_np = [], []
    for i in range(12):
        _, w = wl.make_matmul_inputs(4402 + i, m, 2048, k)
        calls.append(dict(x=xd, w=dev(w), n=2048, independent=True))
        ws_np.append(w)
    calls.insert(9, dict(x=dev(x2), w=dev(w2), n=256, independent=True))
    outs = q2k.MatmulBatch(calls).run()
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    yref2, s2 = oracle.matmul_rows(x2, w2, 256, np.array([0, 100, 255]), threads=ORACLE_THREADS)
    assert_close(outs[9].cpu().numpy()[:, [0, 100, 255]], yref2, s2, TOL_TC, "the call between runs")
    for j, y in enumerate(outs[:9] + outs[10:]):
        yref, s_ = oracle.matmul_rows(x, ws_np[j], 2048, rows, threads=ORACLE_THREADS)
        assert_close(y.cpu().numpy()[:, rows], yref, s_, TOL_TC, f"split run call {j}")


def test_spec_verify_workload_full_in_a_persistent_batch():
    """The spec-verify workload (M=16, N=K=4096) as the bench times it: one of
    many independent projections of one x in a batch, so its call runs in a
    persistent grid.  The workload's own matrix is call 35 of 40 (the second
    grid, on the ready x image); all of its 65536 outputs against the oracle,
    and a sample of call 0's."""
    w_ = wl.WORKLOADS[3]
    inp = wl.make_inputs(w_, with_gather=False)
    rng = np.random.default_rng(4500)
    mats = [wl.random_blocks(rng, w_.n * (w_.k // 256)).reshape(-1) for _ in range(39)]
    mats.insert(35, inp.w)
    xd = dev(inp.x)
    batch = q2k.MatmulBatch([dict(x=xd, w=dev(m), n=w_.n, independent=True) for m in mats])
    assert batch._scratch is not None
    outs = batch.run()
    torch.cuda.synchronize()
    yref, s_ = oracle.matmul(inp.x, inp.w, w_.n, threads=ORACLE_THREADS)
    ratio = assert_close(outs[35].cpu().numpy().astype(np.float64), yref, s_, TOL_TC,
                         "spec-verify in a persistent batch")
    print(f"spec-verify in a persistent batch: max |y - y_ref| / S = {ratio:.3e}")
    rows = np.array([0, 1, 127, 128, 2049, 4095])
    yref0, s0 = oracle.matmul_rows(inp.x, mats[0], w_.n, rows, threads=ORACLE_THREADS)
    assert_close(outs[0].cpu().numpy()[:, rows], yref0, s0, TOL_TC, "call 0 of the batch")


def test_matmul_batch_equals_separate_calls():
    """q2k_matmul_ex_batch (MatmulBatch): GEMV and tensor calls of several
    geometries, the tensor ones sharing a workspace, bit-identical to separate
    q2k.matmul calls; a second run gives the same bits again."""
    specs = [(1, 4096, 4096, dict(independent=True)), (1, 333, 1024, {}), (3, 200, 512, {}),
             (20, 300, 1024, {}), (300, 1000, 512, {}), (300, 1000, 512, {})]
    calls, ref = [], []
    for i, (m, n, k, kw) in enumerate(specs):
        x, w = wl.make_matmul_inputs(3100 + i, m, n, k)
        xd, wd = dev(x), dev(w)
        calls.append(dict(x=xd, w=wd, n=n, **kw))
        ref.append(q2k.matmul(xd, wd, n, **kw))
    # m = 1 calls sharing one x (converted once into the batch scratch), one of
    # them tensor-path, then a call that overwrites that x, then two more on it
    k = 2048
    xs = dev(wl.random_activations(np.random.default_rng(31), 1, k))
    shared = []
    for i, n in enumerate((500, 4096, 77)):
        _, w = wl.make_matmul_inputs(3200 + i, 1, n, k)
        shared.append((n, dev(w)))
    for n, wd in shared:
        calls.append(dict(x=xs, w=wd, n=n, independent=True))
    calls.append(dict(x=xs, w=shared[0][1], n=shared[0][0], path="tensor"))
    x_src = dev(wl.random_activations(np.random.default_rng(32), 1, 256))
    _, w_over = wl.make_matmul_inputs(3300, 1, k, 256)   # writes a fresh x of length k over xs
    calls.append(dict(x=x_src, w=dev(w_over), n=k, out=xs))
    for n, wd in shared[1:]:
        calls.append(dict(x=xs, w=wd, n=n))
    x_keep = xs.clone()
    ref += [q2k.matmul(xs, wd, n, independent=True) for n, wd in shared]
    ref.append(q2k.matmul(xs, shared[0][1], shared[0][0], path="tensor"))
    ref.append(q2k.matmul(x_src, calls[-3]["w"], k))
    ref += [q2k.matmul(ref[-1], wd, n) for n, wd in shared[1:]]
    torch.cuda.synchronize()
    xs.copy_(x_keep)   # the batch starts from the same x
    batch = q2k.MatmulBatch(calls)
    assert batch._scratch is not None  # two groups on xs: before and after the overwrite
    outs = batch.run()
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(outs, ref)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"call {i}"
    first = [o.clone() for o in outs]
    xs.copy_(x_keep)
    batch.run()
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(batch.outs, first)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"rerun call {i}"


def test_tensor_page_run_dense_rows9():
    """Page fn run_dense(9) and the forced-mm variants (rows > 8).

    The page bounds its reduced-precision mm path by 1e-2 absolute at this
    fixture.  The bf16 path here rounds x to 8 significant bits, which at
    input(9) gives up to ~0.05 absolute, so it is held to the relative bf16
    bound 8e-3 * S instead; the fp32 GEMV path (forced) meets the page's 1e-2
    and the fp32 bound.
    """
    w = np.concatenate([wl.page_block(r + 1) for r in range(8)])
    x = wl.page_input(9)
    yref, s = oracle.matmul(x, w, 8)
    for path in ("auto", "tensor"):
        y = run_matmul(x, w, 8, path)
        assert_close(y, yref, s, TOL_TC, f"run_dense(9) {path}")
    y = run_matmul(x, w, 8, "gemv")
    assert np.abs(y - yref).max() <= 1e-2
    assert_close(y, yref, s, TOL_GEMV, "run_dense(9) gemv")


def test_tensor_spec_verify_workload_full():
    w = wl.WORKLOADS[3]
    inp = wl.make_inputs(w, with_gather=False)
    y = run_matmul(inp.x, inp.w, w.n, "auto")
    yref, s = oracle.matmul(inp.x, inp.w, w.n, threads=ORACLE_THREADS)
    ratio = assert_close(y, yref, s, TOL_TC, w.name)
    print(f"{w.name}: max |y - y_ref| / S = {ratio:.3e}")


def test_tensor_prefill_workload_full_every_path():
    """The prefill workload (M=512, N=K=7168) in full, every one of its 3.7 M
    outputs against the oracle: with a workspace (the binding's default), as
    the plain C call q2k_matmul makes it (the library's own scratch), and
    enqueued inside a graph capture (the GEMM converts x itself)."""
    w_ = wl.WORKLOADS[4]
    inp = wl.make_inputs(w_)
    x, w = inp.x, inp.w
    yref, s = oracle.matmul(x, w, w_.n, threads=ORACLE_THREADS)
    xd, wd = dev(x), dev(w)
    lib = q2k.load()
    y_plain = torch.full((w_.m, w_.n), float("nan"), device="cuda")
    p = q2k.MatmulParams(w_.m, w_.n, w_.k, 10)
    st = lib.q2k_matmul(xd.data_ptr(), xd.numel(), wd.data_ptr(), wd.numel(), y_plain.data_ptr(),
                        y_plain.numel(), ctypes.byref(p), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.q2k_last_error().decode()
    results = {"workspace": q2k.matmul(xd, wd, w_.n, path="auto"), "plain C call": y_plain,
               "in-kernel x (capture)": _captured_call(xd, wd, w_.n)}
    torch.cuda.synchronize()
    for name, y in results.items():
        ratio = assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_TC,
                             f"prefill 512x7168x7168 {name}")
        print(f"prefill {name}: max |y - y_ref| / S = {ratio:.3e}")
    assert torch.equal(results["workspace"], results["plain C call"])


def test_tensor_256_row_tiles_sampled_rows():
    """The 256-row tile width at a long N (8192) and short K on sampled weight rows."""
    m, n, k, seed = 512, 8192, 1024, 77
    x, w = wl.make_matmul_inputs(seed, m, n, k)
    y = run_matmul(x, w, n, "auto")
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(n, 40, replace=False), [0, n - 1]]))
    yref, s = oracle.matmul_rows(x, w, n, rows, threads=ORACLE_THREADS)
    ratio = assert_close(y[:, rows], yref, s, TOL_TC, f"m={m} n={n} k={k} sampled")
    print(f"m={m} n={n} k={k}: max |y - y_ref| / S = {ratio:.3e}")


# ------------------------------------------------------------------ properties

@pytest.mark.parametrize("path,m", [("gemv", 1), ("gemv", 5), ("tensor", 40)])
def test_repeated_calls_bit_identical(path, m):
    x, w = wl.make_matmul_inputs(55, m, 300, 2048)
    xd, wd = dev(x), dev(w)
    a = q2k.matmul(xd, wd, 300, path=path)
    b = q2k.matmul(xd, wd, 300, path=path)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("path,m", [("gemv", 3), ("tensor", 20)])
def test_matmul_guard_bands_and_full_overwrite(path, m):
    n, k = 77, 512
    x, w = wl.make_matmul_inputs(66, m, n, k)
    pad = 4096
    buf = torch.full((pad + m * n + pad,), float("nan"), device="cuda")
    y = buf[pad:pad + m * n].view(m, n)
    q2k.matmul(dev(x), dev(w), n, out=y, path=path)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.isnan(host[:pad]).all() and np.isnan(host[-pad:]).all()
    assert not np.isnan(host[pad:-pad]).any()


def test_one_hot_x_gives_the_weight_column():
    n, k = 50, 768
    _, w = wl.make_matmul_inputs(8, 1, n, k)
    W = oracle.dequantize(w).reshape(n, k)
    x = np.zeros((1, k), dtype=np.float32)
    x[0, 300] = 1.0
    y = run_matmul(x, w, n, "gemv")
    assert np.array_equal(y[0], W[:, 300].astype(np.float64))


def test_invalid_arguments_launch_nothing():
    x = torch.zeros((1, 256), device="cuda")
    w = torch.zeros(84 * 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(q2k.InvalidArgument):
        q2k.matmul(x, w[:-1], 8)
    with pytest.raises(q2k.InvalidArgument):
        q2k.matmul(torch.zeros((1, 255), device="cuda"), w, 8)
    lib = q2k.load()
    p = q2k.MatmulParams(1, 8, 256, 10)
    assert lib.q2k_matmul(x.data_ptr(), 256, w.data_ptr(), 672, x.data_ptr(), 8,
                          ctypes.byref(p), None) == 1  # y aliases x


@pytest.mark.parametrize("n,k", [(4096, 4096), (333, 4096), (1000, 1280), (77, 14336)])
def test_const_weights_flag_same_bits(n, k):
    """Q2K_FLAG_CONST_WEIGHTS only moves the weight copies earlier: same bits."""
    x, w = wl.make_matmul_inputs(91 + n, 1, n, k)
    xd, wd = dev(x), dev(w)
    a = q2k.matmul(xd, wd, n)
    b = q2k.matmul(xd, wd, n, const_weights=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    yref, s = oracle.matmul(x, w, n, threads=ORACLE_THREADS)
    assert_close(b.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, f"const n={n} k={k}")


def _captured_call(xd, wd, n):
    """q2k.matmul without a workspace enqueued inside a CUDA graph capture:
    the library then runs the GEMM that converts x itself (no scratch)."""
    s = torch.cuda.Stream()
    out = torch.empty((xd.shape[0], n), dtype=torch.float32, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        q2k.matmul(xd, wd, n, path="tensor", workspace=None, out=out)
    g.replay()
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("m,n,k", [(9, 8, 256), (130, 10000, 256), (300, 1000, 512), (16, 4096, 1024)])
def test_tensor_workspace_and_in_kernel_conversion_agree(m, n, k):
    """With a workspace x is converted by the prepass and the weights-as-A
    kernel runs; a plain call without one uses the library's own scratch for
    the same kernel (bit-identical); inside a graph capture the GEMM converts
    x itself with x as the A operand.  All round x and the weights to bf16 the
    same way; the MMAs differ in orientation, so only the fp32 accumulation
    order may differ."""
    x, w = wl.make_matmul_inputs(3000 + m + n, m, n, k)
    xd, wd = dev(x), dev(w)
    a = _captured_call(xd, wd, n)
    b = q2k.matmul(xd, wd, n, path="tensor")
    c = q2k.matmul(xd, wd, n, path="tensor", workspace=None)
    torch.cuda.synchronize()
    yref, s = oracle.matmul(x, w, n, threads=ORACLE_THREADS)
    ya = a.cpu().numpy().astype(np.float64)
    yb = b.cpu().numpy().astype(np.float64)
    yc = c.cpu().numpy().astype(np.float64)
    assert_close(ya, yref, s, TOL_TC, f"in-kernel x m={m} n={n} k={k}")
    assert_close(yb, yref, s, TOL_TC, f"ws m={m} n={n} k={k}")
    assert np.array_equal(yb, yc), "the plain call's scratch runs the workspace kernel: same bits"
    # same bf16 operands, fp32 sums of k exact products in two orders
    assert np.all(np.abs(ya - yb) <= 1e-5 * s + 1e-30)


def test_plain_calls_on_two_streams_share_the_scratch_safely():
    """Plain (no-workspace) tensor calls on two streams at once: the library's
    scratch is handed from one to the next on the GPU, so both are correct."""
    m, n, k = 300, 2048, 2048
    x1, w1 = wl.make_matmul_inputs(4101, m, n, k)
    x2, w2 = wl.make_matmul_inputs(4102, m, n, k)
    d = [(dev(x1), dev(w1)), (dev(x2), dev(w2))]
    want = [q2k.matmul(xd, wd, n, path="tensor") for xd, wd in d]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    torch.cuda.synchronize()
    for rep in range(6):
        for i, st in enumerate(streams):
            with torch.cuda.stream(st):
                outs[i].append(q2k.matmul(d[i][0], d[i][1], n, path="tensor", workspace=None))
    torch.cuda.synchronize()
    for i in range(2):
        for y in outs[i]:
            assert torch.equal(y, want[i])


def test_plain_call_beyond_the_scratch_converts_x_in_kernel():
    """An x image larger than the library's 32 MiB scratch (m = 4096, k = 4096:
    32 MiB + padding) falls back to the GEMM that converts x itself."""
    m, n, k = 4224, 136, 4096
    x, w = wl.make_matmul_inputs(4103, m, n, k)
    y = q2k.matmul(dev(x), dev(w), n, path="tensor", workspace=None)
    torch.cuda.synchronize()
    yref, s = oracle.matmul(x, w, n, threads=ORACLE_THREADS)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_TC, "beyond scratch")


@pytest.mark.parametrize("n,k", [(4096, 4096), (333, 4096), (14336, 4096), (77, 14336)])
def test_independent_flag_same_bits(n, k):
    """Q2K_FLAG_INDEPENDENT only drops the wait before x is read: same bits."""
    x, w = wl.make_matmul_inputs(191 + n, 1, n, k)
    xd, wd = dev(x), dev(w)
    a = q2k.matmul(xd, wd, n)
    b = q2k.matmul(xd, wd, n, independent=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    yref, s = oracle.matmul(x, w, n, threads=ORACLE_THREADS)
    assert_close(b.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, f"indep n={n} k={k}")


def test_independent_calls_complete_in_order_before_a_dependent_one():
    """Back-to-back independent projections of one x, then a dependent call that
    reads all their outputs at once (their concatenation is its x): it must see
    every projection finished, as must the host after a plain synchronize."""
    n_proj, n, k = 6, 1024, 4096
    x, _ = wl.make_matmul_inputs(501, 1, 1, k)
    ws = [wl.make_matmul_inputs(510 + i, 1, n, k)[1] for i in range(n_proj)]
    w_next = wl.make_matmul_inputs(530, 1, 256, n_proj * n)[1]
    xd = dev(x)
    wds = [dev(w) for w in ws]
    wnd = dev(w_next)
    cat = torch.full((1, n_proj * n), float("nan"), device="cuda")
    for rep in range(3):
        cat.fill_(float("nan"))
        for i in range(n_proj):
            q2k.matmul(xd, wds[i], n, out=cat[:, i * n:(i + 1) * n], independent=True)
        z = q2k.matmul(cat, wnd, 256, const_weights=True)
        torch.cuda.synchronize()
        got = cat.cpu().numpy().astype(np.float64)
        for i in range(n_proj):
            yref, s = oracle.matmul(x, ws[i], n, threads=ORACLE_THREADS)
            assert_close(got[:, i * n:(i + 1) * n], yref, s, TOL_GEMV, f"projection {i}")
        zref, s = oracle.matmul(got.astype(np.float32), w_next, 256, threads=ORACLE_THREADS)
        assert_close(z.cpu().numpy().astype(np.float64), zref, s, TOL_GEMV, f"consumer rep {rep}")


@pytest.mark.parametrize("m", [16, 40])
def test_tensor_small_m_flags_same_bits_and_order(m):
    """The small-m tensor path honours Q2K_FLAG_CONST_WEIGHTS and _INDEPENDENT
    (its weight copies, x conversion and y stores start before the wait for
    the kernel before): the same bits as without, and independent calls still
    finish before a dependent consumer of their outputs runs."""
    n_proj, n, k = 5, 1024, 4096
    x = wl.make_matmul_inputs(601 + m, m, 1, k)[0]
    ws = [wl.make_matmul_inputs(610 + i, m, n, k)[1] for i in range(n_proj)]
    w_next = wl.make_matmul_inputs(630, 1, 512, n)[1]
    xd = dev(x)
    wds = [dev(w) for w in ws]
    wnd = dev(w_next)
    base = [q2k.matmul(xd, wd, n, path="tensor") for wd in wds]
    # projection i writes rows i m .. i m + m - 1 of `stack`, which the
    # consumer then reads as its x
    stack = torch.empty((n_proj * m, n), device="cuda")
    for rep in range(3):
        stack.fill_(float("nan"))
        for i in range(n_proj):
            q2k.matmul(xd, wds[i], n, out=stack[i * m:(i + 1) * m], path="tensor",
                       independent=(rep != 1), const_weights=(rep == 1))
        z = q2k.matmul(stack, wnd, 512, path="tensor")
        torch.cuda.synchronize()
        for i in range(n_proj):
            assert torch.equal(stack[i * m:(i + 1) * m], base[i]), f"projection {i}, rep {rep}"
        zref, s = oracle.matmul(stack.cpu().numpy(), w_next, 512, threads=ORACLE_THREADS)
        assert_close(z.cpu().numpy().astype(np.float64), zref, s, TOL_TC, f"consumer rep {rep}")


def test_bounded_wait_times_out_and_reports_without_fault():
    """The bounded wait every kernel uses, run against a barrier nothing completes:
    it gives up after the limit, the host reads the time-out bit, the read clears
    it, and the context keeps working (a matmul right after is still correct)."""
    assert q2k.device_error() == 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    q2k.selftest_wait_timeout(2000)
    t1.record()
    torch.cuda.synchronize()
    waited_ms = t0.elapsed_time(t1)
    assert 1.5 <= waited_ms < 1000.0, waited_ms
    assert q2k.device_error() == 16  # the GEMV time-out bit
    assert q2k.device_error() == 0
    x, w = wl.make_matmul_inputs(77, 1, 256, 1024)
    y = q2k.matmul(dev(x), dev(w), 256)
    yref, s = oracle.matmul(x, w, 256)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, "after time-out")


def test_matmul_batch_graph_replays_the_same_bits():
    """MatmulBatch(graph=True): the first run enqueues and captures, later runs
    replay the graph; every run gives the bits of the plain batch."""
    rng = np.random.default_rng(77)
    k, n = 1024, 384
    x = dev(wl.random_activations(rng, 1, k))
    ws = [dev(wl.random_blocks(rng, n * (k // 256)).reshape(-1)) for _ in range(3)]
    plain = q2k.MatmulBatch([dict(x=x, w=w, n=n, independent=True) for w in ws])
    graphed = q2k.MatmulBatch([dict(x=x, w=w, n=n, independent=True) for w in ws], graph=True)
    want = [o.clone() for o in plain.run()]
    for _ in range(3):
        for o in graphed.outs:
            o.fill_(float("nan"))
        got = graphed.run()
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    # contents updated in place are picked up by the replay
    x.mul_(2.0)
    want2 = [o.clone() for o in plain.run()]
    got2 = graphed.run()
    torch.cuda.synchronize()
    for a, b in zip(got2, want2):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
