"""GPU parity of the batched matrix-vector and expert-routed (mm_id) products.

Each is checked two ways: against the CPU oracle's definition (fp32 path
bound, |y - y_ref| <= 1e-5 * S) and bit for bit against the single m = 1
matmul of the same batch / route, which the pages require of the batched call
(test q2_k_batched_mv_is_byte_identical_to_independent_dispatches) and which
holds here for the routed call too (the same kernel runs per route).
"""

import numpy as np
import pytest

import oracle
import q2k_workloads as wl

torch = pytest.importorskip("torch")
import ggml_q2_quantized_gb300 as q2k  # noqa: E402
from ggml_q2_quantized_gb300 import build as q2k_build  # noqa: E402

pytestmark = pytest.mark.gpu

TOL_GEMV = 1e-5
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


def assert_close(y, yref, s, tol, what):
    err = np.abs(y - yref)
    assert not np.isnan(y).any(), f"{what}: NaN"
    bad = err > tol * s
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs out of tolerance"


def bits_equal(a, b):
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


# ------------------------------------------------------------------ batched mv

def test_batched_mv_page_case_byte_identical():
    """The page's case: 3 batches of 8 rows block(8 b + r + 1), inputs input(3)."""
    batches, n = 3, 8
    w = np.concatenate([wl.page_block(b * n + r + 1) for b in range(batches) for r in range(n)])
    x = wl.page_input(batches)
    wd, xd = dev(w), dev(x)
    y = q2k.matmul_batched_mv(xd, wd, n)
    per = n * 84
    serial = torch.stack([q2k.matmul(xd[b:b + 1], wd[b * per:(b + 1) * per], n)[0]
                          for b in range(batches)])
    torch.cuda.synchronize()
    assert bits_equal(y, serial)
    yref, s = oracle.matmul_batched_mv(x, w, n)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, "page batched")
    assert np.abs(y.cpu().numpy() - yref).max() <= 2e-4   # the page's dense tolerance


@pytest.mark.parametrize("batches,n,k", [
    (5, 333, 512),     # batch strides 55944 B: every other batch's W is 8 bytes off 16
    (4, 1000, 4096),   # aligned strides, several CTAs per batch
    (2, 40, 16640),    # k > 16384: the row-per-warp kernel for every batch
])
def test_batched_mv_random_byte_identical(batches, n, k):
    rng = np.random.default_rng(batches * n + k)
    w = wl.random_blocks(rng, batches * n * (k // 256)).reshape(-1)
    x = wl.random_activations(rng, batches, k)
    wd, xd = dev(w), dev(x)
    y = q2k.matmul_batched_mv(xd, wd, n)
    per = n * (k // 256) * 84
    serial = torch.stack([q2k.matmul(xd[b:b + 1], wd[b * per:(b + 1) * per], n)[0]
                          for b in range(batches)])
    torch.cuda.synchronize()
    assert bits_equal(y, serial)
    yref, s = oracle.matmul_batched_mv(x, w, n, threads=ORACLE_THREADS)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, f"batched {batches}x{n}x{k}")


@pytest.mark.parametrize("offset", [4, 8, 12])
def test_single_matmul_with_w_off_16_byte_boundary(offset):
    """The m = 1 kernel takes any 4-byte-aligned W (head bytes by plain loads)."""
    n, k = 77, 1024
    x, w = wl.make_matmul_inputs(31 + offset, 1, n, k)
    buf = torch.zeros(w.size + 16, dtype=torch.uint8, device="cuda")
    buf[offset:offset + w.size].copy_(dev(w))
    y = q2k.matmul(dev(x), buf[offset:offset + w.size], n)
    torch.cuda.synchronize()
    yref, s = oracle.matmul(x, w, n)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, f"offset {offset}")


# ------------------------------------------------------------------ mm_id

def _expert_case(tokens, top_k, experts, n=8, gap=0):
    parts = []
    for e in range(experts):
        parts.extend(wl.page_block(e * n + r + 1) for r in range(n))
        parts.append(np.full(gap, 0xFF, dtype=np.uint8))
    w = np.concatenate(parts)
    ids = np.array([(3 * t + slot) % experts for t in range(tokens) for slot in range(top_k)],
                   dtype=np.uint32)
    return w, wl.page_input(tokens), ids, n * 84 + gap


def _route_serial(xd, wd, ids, n, k, top_k, stride):
    rows = []
    size = n * (k // 256) * 84
    for r, e in enumerate(ids.tolist()):
        t = r // top_k
        rows.append(q2k.matmul(xd[t:t + 1], wd[e * stride:e * stride + size], n)[0])
    return torch.stack(rows)


@pytest.mark.parametrize("tokens,top_k,experts", [(2, 2, 3), (33, 6, 8)])
def test_matmul_id_page_cases(tokens, top_k, experts):
    """Page fn run_expert (2, 2, 3) and (33, 6, 8)."""
    n = 8
    w, x, ids, stride = _expert_case(tokens, top_k, experts, n)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id(xd, wd, idd, n, experts, top_k)
    serial = _route_serial(xd, wd, ids, n, 256, top_k, stride)
    torch.cuda.synchronize()
    assert bits_equal(y, serial)
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k)
    got = y.cpu().numpy().astype(np.float64)
    assert_close(got, yref, s, TOL_GEMV, f"run_expert({tokens}, {top_k}, {experts})")
    assert np.abs(got - yref).max() <= 2e-4   # the page's tolerance for this case


def test_matmul_id_random_strided_experts():
    """Larger experts, an expert stride 20 bytes past the matrix (so experts sit
    at different offsets from a 16-byte boundary), random ids."""
    tokens, top_k, experts, n, k = 16, 4, 8, 512, 2048
    rng = np.random.default_rng(5)
    size = n * (k // 256) * 84
    stride = size + 20
    w = np.zeros((experts - 1) * stride + size, dtype=np.uint8)
    for e in range(experts):
        w[e * stride:e * stride + size] = wl.random_blocks(rng, n * (k // 256)).reshape(-1)
    x = wl.random_activations(rng, tokens, k)
    ids = rng.integers(0, experts, tokens * top_k).astype(np.uint32)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id(xd, wd, idd, n, experts, top_k, expert_stride=stride)
    serial = _route_serial(xd, wd, ids, n, k, top_k, stride)
    torch.cuda.synchronize()
    assert bits_equal(y, serial)
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k, threads=ORACLE_THREADS)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, "random mm_id")


def test_matmul_id_bad_id_gives_zero_row_and_count():
    tokens, top_k, experts, n = 4, 2, 3, 8
    w, x, ids, stride = _expert_case(tokens, top_k, experts, n)
    bad = ids.copy()
    bad[5] = experts          # out of range
    bad[6] = 0xFFFFFFFF       # far out of range
    wd, xd, idd = dev(w), dev(x), dev(bad.view(np.int32))
    with pytest.raises(q2k.InvalidArgument):
        q2k.matmul_id(xd, wd, idd, n, experts, top_k)
    y, count = q2k.matmul_id(xd, wd, idd, n, experts, top_k, check=False)
    torch.cuda.synchronize()
    assert int(count.item()) == 2
    got = y.cpu().numpy()
    assert (got[5] == 0).all() and (got[6] == 0).all()
    good = [r for r in range(tokens * top_k) if r not in (5, 6)]
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k)
    assert_close(got[good].astype(np.float64), yref[good], s[good], TOL_GEMV, "good routes")


def test_matmul_id_slotted_equals_flattened_page_case():
    """Page test q2_k_slotted_down_mm_is_byte_identical_to_flattened_rows:
    33 tokens x top_k 6 routes, 8 experts, input(198) as [33, 6, 256]."""
    tokens, top_k, experts, n = 33, 6, 8, 8
    w, _, ids, stride = _expert_case(tokens, top_k, experts, n)
    x = wl.page_input(tokens * top_k)
    wd, idd = dev(w), dev(ids.view(np.int32))
    xd = dev(x)
    slotted = q2k.matmul_id_slotted(xd.view(tokens, top_k, 256), wd, idd.view(tokens, top_k), n,
                                    experts)
    flat = q2k.matmul_id(xd, wd, idd, n, experts, 1)
    torch.cuda.synchronize()
    assert bits_equal(slotted.view(-1, n), flat)
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k, slotted=True)
    got = slotted.view(-1, n).cpu().numpy().astype(np.float64)
    assert_close(got, yref, s, TOL_GEMV, "slotted")
    assert np.abs(got - yref).max() <= 2e-4


def test_matmul_id_pair_page_case_and_distinct_weights():
    """Page fn run_expert(33, 6, 8, force_mm): both weight sets the same, both
    outputs agree bit for bit; then distinct sets, each equal to its own call."""
    tokens, top_k, experts, n = 33, 6, 8, 8
    w, x, ids, stride = _expert_case(tokens, top_k, experts, n)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    ya, yb = q2k.matmul_id_pair(xd, wd, wd, idd, n, experts, top_k)
    single = q2k.matmul_id(xd, wd, idd, n, experts, top_k)
    torch.cuda.synchronize()
    assert bits_equal(ya, yb) and bits_equal(ya, single)
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k)
    assert np.abs(ya.cpu().numpy().astype(np.float64) - yref).max() <= 1e-2  # the page's mm bound
    assert_close(ya.cpu().numpy().astype(np.float64), yref, s, TOL_GEMV, "pair a")
    # distinct second set: experts drawn at random, stride with a gap
    rng = np.random.default_rng(77)
    w2 = np.concatenate([wl.random_blocks(rng, n) for _ in range(experts)])
    ya, yb = q2k.matmul_id_pair(xd, wd, dev(w2), idd, n, experts, top_k)
    sb = q2k.matmul_id(xd, dev(w2), idd, n, experts, top_k)
    torch.cuda.synchronize()
    assert bits_equal(ya, single) and bits_equal(yb, sb)
    yref2, s2 = oracle.matmul_id(x, w2, ids, n, experts, n * 84, top_k)
    assert_close(yb.cpu().numpy().astype(np.float64), yref2, s2, TOL_GEMV, "pair b")


def test_matmul_id_pair_counts_bad_ids_per_product():
    tokens, top_k, experts, n = 3, 2, 3, 8
    w, x, ids, _ = _expert_case(tokens, top_k, experts, n)
    bad = ids.copy()
    bad[1] = 7
    ya, yb, count = q2k.matmul_id_pair(dev(x), dev(w), dev(w), dev(bad.view(np.int32)), n, experts,
                                       top_k, check=False)
    torch.cuda.synchronize()
    assert int(count.item()) == 2
    assert (ya[1] == 0).all() and (yb[1] == 0).all()


def test_x_planes_scratch_gives_the_same_bits():
    """Batched and routed calls with x converted once per row (the default
    scratch) and per CTA (scratch=None) give identical results."""
    rng = np.random.default_rng(9)
    batches, n, k = 4, 700, 4096
    w = wl.random_blocks(rng, batches * n * (k // 256)).reshape(-1)
    x = wl.random_activations(rng, batches, k)
    wd, xd = dev(w), dev(x)
    a = q2k.matmul_batched_mv(xd, wd, n, scratch="auto")
    b = q2k.matmul_batched_mv(xd, wd, n)
    tokens, top_k, experts, ne = 3, 4, 6, 512
    we = wl.random_blocks(rng, experts * ne * (k // 256)).reshape(-1)
    ids = rng.integers(0, experts, tokens * top_k).astype(np.uint32)
    xt = dev(wl.random_activations(rng, tokens, k))
    wed, idd = dev(we), dev(ids.view(np.int32))
    c = q2k.matmul_id(xt, wed, idd, ne, experts, top_k)
    d = q2k.matmul_id(xt, wed, idd, ne, experts, top_k, scratch=None)
    torch.cuda.synchronize()
    assert bits_equal(a, b) and bits_equal(c, d)


# ------------------------------------------------------- mm_id on tensor cores

TOL_TC = 8e-3   # bf16 operands, fp32 accumulation: as the dense tensor path


def _tc_case(rng, tokens, top_k, experts, n, k, stride_pad=0, ids=None):
    size = n * (k // 256) * 84
    stride = size + stride_pad
    w = np.zeros((experts - 1) * stride + size, dtype=np.uint8)
    for e in range(experts):
        w[e * stride:e * stride + size] = wl.random_blocks(rng, n * (k // 256)).reshape(-1)
    x = wl.random_activations(rng, tokens, k)
    if ids is None:
        ids = rng.integers(0, experts, tokens * top_k).astype(np.uint32)
    return w, x, ids, stride


def test_matmul_id_tensor_page_case():
    """Page fn run_expert(33, 6, 8) with force_mm: the matrix path.

    The page holds its reduced-precision mm_id to 1e-2 absolute; the bf16
    operands here round x to 8 significant bits (up to ~0.07 absolute at this
    fixture, as on the dense run_dense(9) case), so the path is held to the
    relative bf16 bound 8e-3 * S; the GEMV path meets the page's 2e-4."""
    tokens, top_k, experts, n = 33, 6, 8, 8
    w, x, ids, stride = _expert_case(tokens, top_k, experts, n)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k, path="tensor")
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k)
    got = y.cpu().numpy().astype(np.float64)
    assert_close(got, yref, s, TOL_TC, "tensor run_expert(33, 6, 8)")
    # auto takes the matrix path above 32 tokens
    ya = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k)
    torch.cuda.synchronize()
    assert bits_equal(ya, y)


@pytest.mark.parametrize("tokens,top_k,experts,n,k,pad", [
    (80, 6, 8, 320, 1024, 0),       # ragged n (2.5 weight tiles), TMA weights
    (70, 4, 16, 200, 512, 0),       # rows not a multiple of 1024 bytes: no TMA view
    (48, 8, 6, 256, 2048, 2 * 84 * 8),  # stride a whole number of rows past the matrix
    (40, 2, 5, 136, 1024, 20),      # stride off the row size: per-expert offsets, no TMA
])
def test_matmul_id_tensor_random(tokens, top_k, experts, n, k, pad):
    rng = np.random.default_rng(tokens * 7 + k)
    w, x, ids, stride = _tc_case(rng, tokens, top_k, experts, n, k, pad)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k, path="tensor", expert_stride=stride)
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k, threads=ORACLE_THREADS)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_TC,
                 f"tensor mm_id {tokens}x{top_k} of {experts}, {n}x{k}")


def test_matmul_id_tensor_skewed_routes():
    """One expert takes 300 routes (three x tiles, the last ragged), several
    take none, the rest one each: the tile table's edge cases."""
    tokens, top_k, experts, n, k = 150, 2, 12, 256, 1024
    ids = np.full(tokens * top_k, 3, dtype=np.uint32)
    ids[::37] = 7
    ids[5] = 11
    ids[8] = 0
    rng = np.random.default_rng(9)
    w, x, ids, stride = _tc_case(rng, tokens, top_k, experts, n, k, ids=ids)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k, path="tensor")
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k, threads=ORACLE_THREADS)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_TC, "skewed tensor mm_id")


def test_matmul_id_tensor_slotted_and_bad_ids():
    tokens, top_k, experts, n, k = 40, 4, 6, 256, 1024
    rng = np.random.default_rng(21)
    w, _, ids, stride = _tc_case(rng, tokens, top_k, experts, n, k)
    x = wl.random_activations(rng, tokens * top_k, k).reshape(tokens, top_k, k)
    bad = ids.copy()
    bad[3] = experts
    bad[77] = 0xFFFFFFFF
    wd, xd, idd = dev(w), dev(x), dev(bad.view(np.int32))
    y, count = q2k.matmul_id_ex(xd, wd, idd, n, experts, path="tensor", slotted=True, check=False)
    torch.cuda.synchronize()
    assert int(count.item()) == 2
    got = y.cpu().numpy().reshape(tokens * top_k, n)
    assert (got[3] == 0).all() and (got[77] == 0).all()
    yref, s = oracle.matmul_id(x.reshape(tokens * top_k, k), w, ids, n, experts, stride, 1,
                               threads=ORACLE_THREADS)
    good = [r for r in range(tokens * top_k) if r not in (3, 77)]
    assert_close(got[good].astype(np.float64), yref[good], s[good], TOL_TC, "slotted tensor mm_id")


def test_matmul_id_tensor_moe_prefill_sampled():
    """The MoE layer's prefill shape (512 tokens, top-8 of 64 experts of
    2048 x 7168): sampled routes against the oracle."""
    tokens, top_k, experts, n, k = 512, 8, 64, 2048, 7168
    rng = np.random.default_rng(31)
    w, x, ids, stride = _tc_case(rng, tokens, top_k, experts, n, k)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k, path="tensor").cpu().numpy()
    routes = rng.choice(tokens * top_k, 12, replace=False)
    size = n * (k // 256) * 84
    for r in routes.tolist():
        e = int(ids[r])
        yref, s = oracle.matmul(x[r // top_k:r // top_k + 1], w[e * stride:e * stride + size], n)
        assert_close(y[r:r + 1].astype(np.float64), yref, s, TOL_TC, f"route {r}")


def test_matmul_id_pair_tensor_shares_routing():
    """Page fn run_expert with force_mm runs the pair on its matrix path: here
    routing and the x gather run once and each weight set's GEMM reads the same
    tiles, so each output equals its own tensor-path call bit for bit."""
    tokens, top_k, experts, n, k = 48, 6, 8, 320, 1024
    rng = np.random.default_rng(41)
    wa, x, ids, stride = _tc_case(rng, tokens, top_k, experts, n, k)
    wb, _, _, _ = _tc_case(rng, tokens, top_k, experts, n, k, ids=ids)
    bad = ids.copy()
    bad[10] = experts + 3
    xd, idd = dev(x), dev(bad.view(np.int32))
    wad, wbd = dev(wa), dev(wb)
    ya, yb, count = q2k.matmul_id_pair(xd, wad, wbd, idd, n, experts, top_k, path="tensor",
                                       check=False)
    sa, ca = q2k.matmul_id_ex(xd, wad, idd, n, experts, top_k, path="tensor", check=False)
    sb, cb = q2k.matmul_id_ex(xd, wbd, idd, n, experts, top_k, path="tensor", check=False)
    torch.cuda.synchronize()
    assert int(count.item()) == 2 and int(ca.item()) == 1 and int(cb.item()) == 1
    assert bits_equal(ya, sa) and bits_equal(yb, sb)
    good = [r for r in range(tokens * top_k) if r != 10]
    for y, w in ((ya, wa), (yb, wb)):
        got = y.cpu().numpy()
        assert (got[10] == 0).all()
        yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k, threads=ORACLE_THREADS)
        assert_close(got[good].astype(np.float64), yref[good], s[good], TOL_TC, "pair tensor")


@pytest.mark.parametrize("experts,tokens,top_k", [(4096, 40, 2), (1, 70, 1), (3, 33, 3)])
def test_matmul_id_tensor_expert_counts(experts, tokens, top_k):
    """The routing kernel's scan at its limits: 4096 experts (4 per scan thread,
    most empty), a single expert (every route in one expert's tiles), and auto
    at 33 tokens (the first count the matrix path takes)."""
    n, k = 8 if experts > 8 else 136, 256 if experts > 8 else 1024
    rng = np.random.default_rng(experts + tokens)
    w, x, ids, stride = _tc_case(rng, tokens, top_k, experts, n, k)
    if experts == 4096:
        ids = rng.choice(experts, tokens * top_k, replace=False).astype(np.uint32)
    wd, xd, idd = dev(w), dev(x), dev(ids.view(np.int32))
    y = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k, path="auto")
    yt = q2k.matmul_id_ex(xd, wd, idd, n, experts, top_k, path="tensor")
    torch.cuda.synchronize()
    assert bits_equal(y, yt)   # more than 32 tokens: auto is the tensor path
    yref, s = oracle.matmul_id(x, w, ids, n, experts, stride, top_k, threads=ORACLE_THREADS)
    assert_close(y.cpu().numpy().astype(np.float64), yref, s, TOL_TC,
                 f"tensor mm_id, {experts} experts")
