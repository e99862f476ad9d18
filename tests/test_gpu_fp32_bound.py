"""The fp32 path's error bound |y - y_ref| <= 1e-5 * S (S = sum_k |x w|) on
activations chosen to break kernels that round x or factor the block scales.

The GEMV forms each weight exactly as the page's f32 decode (mlx-native page
"tests/deepseek_q2_k.rs", fn reference_dequant: dl*q - ml rounded once) and
accumulates x*w in fp32 along chains of bounded length, so the bound holds for
any finite x whose products stay in the f32 normal range.  These cases put
large values where they add nothing to S:
  - one outlier per 16-weight run (x 1e3, 1e5, 1e7);
  - outliers on weights that are exactly zero in every row, both the plain
    zeros (q = 0 with min nibble 0) and cancelling ones (d = dmin, sc = m,
    q = 1: d*sc*1 - dmin*m = 0);
  - runs mixing 1e-30 and 1, all-zero runs, an all-zero x;
  - heavy-tailed activations with a few channels x100..x1000 (LLM-like);
  - very large |x| (the kernel's rescaled slices).
Each case runs through the m = 1 kernel (plain, const-weights and independent
launches), the batched and routed launches (with and without prepared x), and
the general-m kernel; the worst |y - y_ref| / S is printed.
"""

import zlib

import numpy as np
import pytest

import oracle
import q2k_workloads as wl

torch = pytest.importorskip("torch")
import ggml_q2_quantized_gb300 as q2k  # noqa: E402
from ggml_q2_quantized_gb300 import build as q2k_build  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-5
THREADS = 16


@pytest.fixture(scope="module", autouse=True)
def gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    q2k_build.build()
    q2k.load()
    yield
    assert q2k.device_error() == 0, "a kernel gave up waiting on a barrier"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def ratio(y, yref, s):
    y = np.asarray(y, dtype=np.float64)
    assert not np.isnan(y).any(), "NaN in output"
    err = np.abs(y - yref)
    bad = err > TOL * s
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{bad.sum()} outputs beyond 1e-5*S; first {i}: got {y[i]!r}, "
                             f"want {yref[i]!r}, S={s[i]!r}")
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(s > 0, err / s, 0.0)
    return float(r.max())


# ---- input construction ------------------------------------------------------

def kpos(b, h, j, seg, lane):
    """Weight index of (block, half, shift j, segment, lane) in a row."""
    return 256 * b + 128 * h + 32 * j + 16 * seg + lane


def zero_weight_columns(w, n, k, rng, count, kind):
    """Make `count` weight columns exactly zero in every row; return their k.

    kind "plain": min nibble 0 of the run and code 0 at the lane (w = -0*dmin + 0);
    kind "cancel": dmin = d for the block, scale byte (v << 4) | v for the run,
    code 1 at the lane (w = d*v*1 - d*v = 0 exactly)."""
    B = k // 256
    wb = w.reshape(n, B, 84)
    ks = []
    used = set()
    while len(ks) < count:
        b, h, j, seg, lane = (int(rng.integers(B)), int(rng.integers(2)), int(rng.integers(4)),
                              int(rng.integers(2)), int(rng.integers(16)))
        if (b, h, j, seg) in used:
            continue
        used.add((b, h, j, seg))
        sbyte = 8 * h + 2 * j + seg
        qbyte = 16 + 32 * h + 16 * seg + lane
        if kind == "plain":
            wb[:, b, sbyte] &= 0x0F
            wb[:, b, qbyte] &= np.uint8(~(3 << (2 * j)) & 0xFF)
        else:
            v = int(rng.integers(1, 16))
            wb[:, b, sbyte] = (v << 4) | v
            wb[:, b, 82:84] = wb[:, b, 80:82]
            wb[:, b, qbyte] = (wb[:, b, qbyte] & np.uint8(~(3 << (2 * j)) & 0xFF)) | (1 << (2 * j))
        ks.append(kpos(b, h, j, seg, lane))
    return np.array(ks)


def make_case(name, n, k, seed):
    """(x [1, k] f32, w bytes) for the named adversarial case."""
    rng = np.random.default_rng(seed)
    w = wl.random_blocks(rng, n * (k // 256)).copy()
    x = rng.standard_normal(k).astype(np.float32)
    if name.startswith("outlier_run_"):
        f = float(name.rsplit("_", 1)[1])
        pos = np.arange(0, k, 16) + rng.integers(0, 16, k // 16)
        x[pos] *= np.float32(f)
    elif name in ("zero_w_plain", "zero_w_cancel"):
        ks = zero_weight_columns(w, n, k, rng, max(4, k // 512), name.split("_")[-1])
        x[ks] = np.float32(1e7) * np.where(rng.random(ks.size) < 0.5, -1, 1)
    elif name == "zero_w_tiny_rest":
        # S made only of 1e-30-sized terms; the 1.0s all sit on zero weights
        ks = zero_weight_columns(w, n, k, rng, max(4, k // 512), "plain")
        x = (rng.standard_normal(k) * 1e-30).astype(np.float32)
        x[ks] = 1.0
    elif name == "mix_1e-30_and_1":
        x = np.where(rng.random(k) < 0.5, 1e-30, 1.0).astype(np.float32)
        x *= np.where(rng.random(k) < 0.5, -1, 1).astype(np.float32)
    elif name == "zero_runs":
        runs = rng.choice(k // 16, size=k // 64, replace=False)
        for r in runs:
            x[16 * r:16 * r + 16] = 0.0
    elif name == "all_zero":
        x[:] = 0.0
    elif name == "llm_channels":
        ch = rng.choice(k, size=max(3, k // 1024), replace=False)
        x[ch] *= rng.uniform(100.0, 1000.0, ch.size).astype(np.float32)
    elif name == "huge":
        x *= np.float32(1e30)
        x[rng.integers(k)] = np.float32(1e37)   # x w stays below the f32 maximum
    elif name == "subnormal_scale_mix":
        x *= np.float32(1e-20)
        x[rng.integers(k)] = np.float32(1e20)
    else:
        raise ValueError(name)
    return x.reshape(1, k), w


CASES = ["outlier_run_1e3", "outlier_run_1e5", "outlier_run_1e7", "zero_w_plain", "zero_w_cancel",
         "zero_w_tiny_rest", "mix_1e-30_and_1", "zero_runs", "all_zero", "llm_channels", "huge",
         "subnormal_scale_mix"]


# ---- the m = 1 kernel ---------------------------------------------------------

@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("n,k", [(512, 4096), (300, 14336), (40, 768)])
def test_m1_kernel_bound(case, n, k):
    x, w = make_case(case, n, k, seed=zlib.crc32(f"{case}/{n}/{k}".encode()))
    yref, s = oracle.matmul(x, w, n, threads=THREADS)
    xd, wd = dev(x), dev(w)
    worst = 0.0
    ys = []
    for kw in ({}, {"const_weights": True}, {"independent": True}):
        y = q2k.matmul(xd, wd, n, path="gemv", **kw)
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy())
        worst = max(worst, ratio(ys[-1], yref, s))
    # the flags change scheduling only
    assert all(np.array_equal(ys[0].view(np.uint32), t.view(np.uint32)) for t in ys[1:])
    if case == "all_zero":
        assert not ys[0].any()
    print(f"\n{case} n={n} k={k}: worst |y - y_ref|/S = {worst:.3g}")


@pytest.mark.parametrize("name", ["decode_gemv_4096", "ffn_pair_down"])
@pytest.mark.parametrize("case", ["llm_channels", "outlier_run_1e5", "zero_w_cancel"])
def test_workload_shapes_bound(name, case):
    wk = wl.by_name(name)
    x, w = make_case(case, wk.n, wk.k, seed=17)
    yref, s = oracle.matmul(x, w, wk.n, threads=THREADS)
    y = q2k.matmul(dev(x), dev(w), wk.n, path="gemv", independent=True)
    torch.cuda.synchronize()
    print(f"\n{name} {case}: worst |y - y_ref|/S = {ratio(y.cpu().numpy(), yref, s):.3g}")


# ---- batched, routed, general m ------------------------------------------------

@pytest.mark.parametrize("case", ["outlier_run_1e7", "zero_w_plain", "zero_w_cancel", "llm_channels",
                                  "huge"])
@pytest.mark.parametrize("scratch", [None, "auto"])
def test_batched_and_routed_bound(case, scratch):
    n, k, batches = 256, 4096, 3
    xs, ws = zip(*[make_case(case, n, k, seed=100 + b) for b in range(batches)])
    x = np.concatenate(xs)
    w = np.concatenate(ws)
    yb = q2k.matmul_batched_mv(dev(x), dev(w), n, scratch=scratch)
    torch.cuda.synchronize()
    yb = yb.cpu().numpy()
    for b in range(batches):
        yref, s = oracle.matmul(xs[b], ws[b], n, threads=THREADS)
        ratio(yb[b:b + 1], yref, s)
    # routed: 3 experts, 2 tokens, top-2
    ids = np.array([2, 0, 1, 2], dtype=np.uint32)
    x2 = x[:2].copy()
    yr = q2k.matmul_id(dev(x2), dev(w), dev(ids.view(np.int32)), n, batches, 2, scratch=scratch)
    torch.cuda.synchronize()
    yr = yr.cpu().numpy()
    for r, e in enumerate(ids):
        yref, s = oracle.matmul(x2[r // 2:r // 2 + 1], ws[e], n, threads=THREADS)
        ratio(yr[r:r + 1], yref, s)


@pytest.mark.parametrize("case", ["outlier_run_1e7", "zero_w_cancel", "zero_w_tiny_rest", "huge"])
@pytest.mark.parametrize("m,k", [(3, 4096), (8, 2048), (1, 16640)])
def test_general_m_kernel_bound(case, m, k):
    """m = 2..8, and m = 1 with k above the m = 1 kernel's limit: gemv_rows_kernel."""
    n = 64
    x0, w = make_case(case, n, k, seed=300 + m)
    # every row keeps the case's structure (outliers on the same columns)
    x = (x0 * np.random.default_rng(m).uniform(0.5, 1.5, (m, k))).astype(np.float32)
    yref, s = oracle.matmul(x, w, n, threads=THREADS)
    y = q2k.matmul(dev(x), dev(w), n, path="gemv")
    torch.cuda.synchronize()
    print(f"\n{case} m={m} k={k}: worst |y - y_ref|/S = {ratio(y.cpu().numpy(), yref, s):.3g}")
