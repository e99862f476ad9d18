"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with what the mlx-native test page "tests/deepseek_q2_k.rs" or
plain mathematics fixes.  ``test_oracle_pins.py`` runs them on the oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with one planted
mistake each and requires that some pin fails for every copy.

Sources of truth used here (none of them is the oracle's own code path):
  * numpy's binary16 -> binary32 conversion (all 65536 bit patterns);
  * values decoded by hand from the page's ``block(5)`` fixture
    (``golden/page_block5_hand_values.txt``, with the derivation);
  * the element position closed form k = 128 half + 32 j + 16 segment + lane
    (shift = 2 j) and scale index 8 half + 2 j + segment, read off the page's
    loop nest, checked with one-hot blocks;
  * exact rational arithmetic (``fractions.Fraction``) for d*sc*q - dmin*m;
  * ``math.fsum`` and exact dyadic arithmetic for the matmul;
  * the page's own assertions (sign mix, malformed-buffer and bad-id errors,
    the gather test, the 2e-4 tolerance of its dense test).
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import q2k_workloads as wl
from oracle import OracleError

QK_K = 256
BLOCK_BYTES = 84
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f16_bits(value: float) -> int:
    return int(np.array([value], dtype="<f2").view(np.uint16)[0])


def make_block(scales, qs, d_bits: int, dmin_bits: int) -> np.ndarray:
    b = np.zeros(BLOCK_BYTES, dtype=np.uint8)
    b[0:16] = np.asarray(scales, dtype=np.uint8)
    b[16:80] = np.asarray(qs, dtype=np.uint8)
    b[80] = d_bits & 0xFF
    b[81] = d_bits >> 8
    b[82] = dmin_bits & 0xFF
    b[83] = dmin_bits >> 8
    return b


def position(half: int, j: int, segment: int, lane: int) -> int:
    return 128 * half + 32 * j + 16 * segment + lane


def scale_index_of(k: int) -> int:
    half, rem = divmod(k, 128)
    j, rem = divmod(rem, 32)
    segment = rem // 16
    return 8 * half + 2 * j + segment


def quant_byte_of(k: int) -> int:
    half, rem = divmod(k, 128)
    rem %= 32
    segment, lane = divmod(rem, 16)
    return 32 * half + 16 * segment + lane


def f16_value(bits: int) -> Fraction:
    return Fraction(float(np.array([bits], dtype=np.uint16).view("<f2")[0]))


# --------------------------------------------------------------------- decode

def pin_f16_all_patterns(o):
    """Every binary16 pattern decodes like numpy's float16 -> float32 cast."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = o.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan), "NaN patterns differ"
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32)), \
        "binary16 decode differs from numpy"


def pin_block5_hand_values(o):
    """Hand-decoded values of the page fixture block(5)."""
    out = o.dequant_block(wl.page_block(5))
    with open(os.path.join(GOLDEN, "page_block5_hand_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for k, v in rows:
        assert out[int(k)] == np.float32(float(v)), f"block(5)[{k}] = {out[int(k)]}, want {v}"


def pin_block5_signs(o):
    """Page test q2_k_host_decode_matches_all_256_canonical_values: both signs occur."""
    out = o.dequant_block(wl.page_block(5))
    assert out.size == QK_K
    assert (out < 0).any() and (out > 0).any()


def pin_one_hot_positions(o):
    """A single q=1 field lands at the closed-form position, all else is zero."""
    one, zero = f16_bits(1.0), f16_bits(0.0)
    for byte in range(64):
        half, rem = divmod(byte, 32)
        segment, lane = divmod(rem, 16)
        for j in range(4):
            qs = np.zeros(64, dtype=np.uint8)
            qs[byte] = 1 << (2 * j)
            out = o.dequant_block(make_block(np.ones(16), qs, one, zero))
            want = np.zeros(QK_K, dtype=np.float32)
            want[position(half, j, segment, lane)] = 1.0
            assert np.array_equal(out, want), f"one-hot quant byte {byte} shift {2 * j}"


def pin_scale_index(o):
    """With q = 1 everywhere, d = 1, dmin = 0 and scale byte s = s, w[k] = scale index."""
    scales = np.arange(16, dtype=np.uint8)
    out = o.dequant_block(make_block(scales, np.full(64, 0x55), f16_bits(1.0), f16_bits(0.0)))
    want = np.array([scale_index_of(k) for k in range(QK_K)], dtype=np.float32)
    assert np.array_equal(out, want), "scale index mapping"


def pin_min_index(o):
    """With q = 0, d = dmin = 1 and high nibble s in scale byte s, w[k] = -scale index."""
    scales = (np.arange(16, dtype=np.uint8) << 4).astype(np.uint8)
    out = o.dequant_block(make_block(scales, np.zeros(64), f16_bits(1.0), f16_bits(1.0)))
    want = -np.array([scale_index_of(k) for k in range(QK_K)], dtype=np.float32)
    assert np.array_equal(out, want), "min nibble mapping"


def pin_exact_all_combinations(o, seed: int = 11):
    """All (scale, min, q) combinations equal RN_f32(d*sc*q - dmin*m) computed exactly.

    Every product is exact in f32 (d has an 11-bit significand, sc*q < 64), so
    the page's separately rounded f32 steps give the exactly rounded value.
    """
    rng = np.random.default_rng(seed)
    ds = [f16_bits(v) for v in rng.uniform(0.001, 0.05, 3)]
    ds += [0x0001, 0x03FF, 0x7BFF, f16_bits(1.0)]  # smallest subnormal, largest subnormal, max
    dmins = [f16_bits(v) for v in rng.uniform(0.001, 0.05, 3)]
    dmins += [0x0400, 0x0001, 0x7BFF, f16_bits(0.5)]
    combos = [(sc, m) for m in range(16) for sc in range(16)]
    for d_bits, dmin_bits in zip(ds, dmins):
        d, dmin = f16_value(d_bits), f16_value(dmin_bits)
        for start in range(0, 256, 16):
            group = combos[start:start + 16]
            scales = [(m << 4) | sc for sc, m in group]
            qs = np.zeros(64, dtype=np.uint8)
            for byte in range(64):
                qs[byte] = sum(((byte + j) % 4) << (2 * j) for j in range(4))
            out = o.dequant_block(make_block(scales, qs, d_bits, dmin_bits))
            for k in range(QK_K):
                sc, m = group[scale_index_of(k)]
                q = (int(qs[quant_byte_of(k)]) >> (2 * ((k % 128) // 32))) & 3
                exact = d * sc * q - dmin * m
                want = np.float32(float(exact))
                assert out[k] == want, f"k={k} sc={sc} m={m} q={q}: {out[k]} != {want}"


def pin_zero_quants_constant(o, seed: int = 12):
    """All-zero quants: every 16-lane segment is the constant -dmin*m."""
    rng = np.random.default_rng(seed)
    scales = rng.integers(0, 256, 16)
    d_bits, dmin_bits = f16_bits(0.0371), f16_bits(0.0123)
    out = o.dequant_block(make_block(scales, np.zeros(64), d_bits, dmin_bits))
    dmin = f16_value(dmin_bits)
    for k in range(QK_K):
        m = int(scales[scale_index_of(k)]) >> 4
        assert out[k] == np.float32(float(-dmin * m)), f"k={k}"


def pin_zero_scale_nibble(o, seed: int = 13):
    """Scale nibble 0: the segment is -dmin*m whatever the quants are."""
    rng = np.random.default_rng(seed)
    scales = (rng.integers(0, 16, 16) << 4).astype(np.uint8)
    qs = rng.integers(0, 256, 64)
    out = o.dequant_block(make_block(scales, qs, f16_bits(0.02), f16_bits(0.03)))
    dmin = f16_value(f16_bits(0.03))
    for k in range(QK_K):
        assert out[k] == np.float32(float(-dmin * (int(scales[scale_index_of(k)]) >> 4)))


def pin_zero_d_dmin(o, seed: int = 14):
    rng = np.random.default_rng(seed)
    out = o.dequant_block(make_block(rng.integers(0, 256, 16), rng.integers(0, 256, 64), 0, 0))
    assert np.array_equal(out, np.zeros(QK_K, dtype=np.float32))


def pin_malformed_buffers(o):
    """Page test q2_k_host_decode_rejects_malformed_buffers (83 bytes, 255 floats)."""
    b = wl.page_block(1)
    for args in ((b[:83], None), (b, 255), (b, 257)):
        try:
            o.dequantize(*args)
        except OracleError:
            continue
        raise AssertionError(f"malformed buffer accepted: {args[0].size} bytes, n_out={args[1]}")
    assert o.dequantize(b).size == QK_K


def pin_gather_page(o):
    """Page gather test: vocab 3 of rows block(row+2), ids [2, 0]; id = vocab is an error."""
    table = np.concatenate([wl.page_block(r + 2) for r in range(3)])
    out = o.gather(table, 3, QK_K, [2, 0])
    assert np.array_equal(out[0], o.dequant_block(wl.page_block(4)))
    assert np.array_equal(out[1], o.dequant_block(wl.page_block(2)))
    try:
        o.gather(table, 3, QK_K, [2, 3])
    except OracleError:
        return
    raise AssertionError("id == vocab accepted")


# --------------------------------------------------------------------- matmul

def _decoded_rows(o, w, n, k):
    return o.dequantize(w).reshape(n, k)


def pin_matmul_one_hot(o, seed: int = 21):
    """x[m] = e_{k_m} gives y[m, r] = w[r, k_m] exactly (rows and blocks indexed right)."""
    M, N, K = 3, 5, 768
    _, w = wl.make_matmul_inputs(seed, 1, N, K)
    W = _decoded_rows(o, w, N, K)
    ks = [7, 300, 767]
    x = np.zeros((M, K), dtype=np.float32)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    y, s = o.matmul(x, w, N)
    for m, k in enumerate(ks):
        assert np.array_equal(y[m], W[:, k].astype(np.float64)), f"one-hot row {m}"
        assert np.array_equal(s[m], np.abs(W[:, k]).astype(np.float64))


def pin_matmul_linearity(o, seed: int = 22):
    """y(2 x1 + x2) = 2 y(x1) + y(x2) exactly for dyadic x (all f64 sums exact)."""
    M, N, K = 2, 4, 512
    rng = np.random.default_rng(seed)
    _, w = wl.make_matmul_inputs(seed, 1, N, K)
    x1 = (rng.integers(-16, 17, (M, K)) / 8).astype(np.float32)
    x2 = (rng.integers(-16, 17, (M, K)) / 8).astype(np.float32)
    y1, _ = o.matmul(x1, w, N)
    y2, _ = o.matmul(x2, w, N)
    y3, _ = o.matmul((2 * x1 + x2).astype(np.float32), w, N)
    assert np.array_equal(y3, 2 * y1 + y2)


def pin_matmul_fsum(o, seed: int = 23):
    """Against math.fsum of the exact f64 products of the decoded rows."""
    M, N, K = 3, 4, 512
    x, w = wl.make_matmul_inputs(seed, M, N, K)
    W = _decoded_rows(o, w, N, K).astype(np.float64)
    y, s = o.matmul(x, w, N)
    for m in range(M):
        for r in range(N):
            terms = x[m].astype(np.float64) * W[r]
            ref = math.fsum(terms)
            ref_abs = math.fsum(np.abs(terms))
            assert abs(y[m, r] - ref) <= 1e-12 * ref_abs, f"y[{m},{r}]"
            assert abs(s[m, r] - ref_abs) <= 1e-12 * ref_abs, f"s_abs[{m},{r}]"


def pin_run_dense_page(o):
    """Page fn run_dense(1): 8 rows block(r+1), x = input(1), within its 2e-4 of cpu_dot."""
    n = 8
    w = np.concatenate([wl.page_block(r + 1) for r in range(n)])
    x = wl.page_input(1)
    y, _ = o.matmul(x, w, n)
    for r in range(n):
        dec = o.dequant_block(wl.page_block(r + 1))
        acc = np.float32(0.0)
        for a, b in zip(dec, x[0]):
            acc = np.float32(acc + np.float32(a * b))
        assert abs(y[0, r] - float(acc)) <= 2e-4, f"row {r}"


def _fsum_dot(x_row, w_row):
    terms = x_row.astype(np.float64) * w_row.astype(np.float64)
    return math.fsum(terms), math.fsum(np.abs(terms))


def pin_batched_mv_page(o):
    """Page test q2_k_batched_mv_is_byte_identical_to_independent_dispatches:
    3 batches of 8 rows block(8 b + r + 1), inputs input(3); batch b is its own
    matrix times its own input row (math.fsum of the decoded products)."""
    batches, n = 3, 8
    w = np.concatenate([wl.page_block(b * n + r + 1) for b in range(batches) for r in range(n)])
    x = wl.page_input(batches)
    y, s = o.matmul_batched_mv(x, w, n)
    assert y.shape == (batches, n)
    for b in range(batches):
        for r in range(n):
            ref, ref_abs = _fsum_dot(x[b], o.dequant_block(wl.page_block(b * n + r + 1)))
            assert abs(y[b, r] - ref) <= 1e-12 * ref_abs, f"batch {b} row {r}"
            assert abs(s[b, r] - ref_abs) <= 1e-12 * ref_abs


def _expert_fixture(tokens, top_k, experts, n=8, gap=0):
    """Page fn run_expert: expert e's row r is block(e n + r + 1), x = input(tokens),
    ids[t top_k + slot] = (3 t + slot) mod experts.  ``gap`` bytes of 0xFF between
    experts make expert_stride larger than one expert's matrix."""
    parts = []
    for e in range(experts):
        parts.extend(wl.page_block(e * n + r + 1) for r in range(n))
        parts.append(np.full(gap, 0xFF, dtype=np.uint8))
    w = np.concatenate(parts)
    ids = np.array([(3 * t + slot) % experts for t in range(tokens) for slot in range(top_k)],
                   dtype=np.uint32)
    return w, wl.page_input(tokens), ids, n * BLOCK_BYTES + gap


def pin_matmul_id_page(o):
    """Page fn run_expert(2, 2, 3) and run_expert(33, 6, 8): route r (token-major)
    is expert ids[r]'s rows times token r // top_k's input."""
    for tokens, top_k, experts in ((2, 2, 3), (33, 6, 8)):
        n = 8
        w, x, ids, stride = _expert_fixture(tokens, top_k, experts, n)
        y, _ = o.matmul_id(x, w, ids, n, experts, stride, top_k)
        assert y.shape == (tokens * top_k, n)
        for r in range(tokens * top_k):
            t, e = r // top_k, int(ids[r])
            for row in range(n):
                ref, ref_abs = _fsum_dot(x[t], o.dequant_block(wl.page_block(e * n + row + 1)))
                assert abs(y[r, row] - ref) <= 1e-12 * ref_abs, f"route {r} row {row}"


def pin_matmul_id_stride_and_bad_id(o):
    """Experts are expert_stride bytes apart (not packed), and an id >= n_experts
    is an error (the pages reject bad ids)."""
    tokens, top_k, experts, n = 3, 2, 4, 8
    w, x, ids, stride = _expert_fixture(tokens, top_k, experts, n, gap=52)
    y, _ = o.matmul_id(x, w, ids, n, experts, stride, top_k)
    for r in range(tokens * top_k):
        t, e = r // top_k, int(ids[r])
        ref, ref_abs = _fsum_dot(x[t], o.dequant_block(wl.page_block(e * n + n)))
        assert abs(y[r, n - 1] - ref) <= 1e-12 * ref_abs, f"route {r}"
    bad = ids.copy()
    bad[3] = experts
    try:
        o.matmul_id(x, w, bad, n, experts, stride, top_k)
    except OracleError:
        pass
    else:
        raise AssertionError("an expert id >= n_experts was accepted")


def pin_matmul_id_slotted_page(o):
    """Page test q2_k_slotted_down_mm_is_byte_identical_to_flattened_rows: 33 tokens,
    top_k 6, 8 experts, one input row per route (input(198)); the slotted product
    equals the flattened one (n_tokens 198, top_k 1), and route r is expert ids[r]
    times input row r."""
    tokens, top_k, experts, n = 33, 6, 8, 8
    w, _, ids, stride = _expert_fixture(tokens, top_k, experts, n)
    x = wl.page_input(tokens * top_k)
    ys, _ = o.matmul_id(x, w, ids, n, experts, stride, top_k, slotted=True)
    yf, _ = o.matmul_id(x, w, ids, n, experts, stride, 1)
    assert np.array_equal(ys, yf)
    for r in (0, 5, 6, 100, 197):
        e = int(ids[r])
        for row in (0, n - 1):
            ref, ref_abs = _fsum_dot(x[r], o.dequant_block(wl.page_block(e * n + row + 1)))
            assert abs(ys[r, row] - ref) <= 1e-12 * ref_abs, f"route {r} row {row}"


ALL_PINS = [
    pin_f16_all_patterns,
    pin_block5_hand_values,
    pin_block5_signs,
    pin_one_hot_positions,
    pin_scale_index,
    pin_min_index,
    pin_exact_all_combinations,
    pin_zero_quants_constant,
    pin_zero_scale_nibble,
    pin_zero_d_dmin,
    pin_malformed_buffers,
    pin_gather_page,
    pin_matmul_one_hot,
    pin_matmul_linearity,
    pin_matmul_fsum,
    pin_run_dense_page,
    pin_batched_mv_page,
    pin_matmul_id_page,
    pin_matmul_id_stride_and_bad_id,
    pin_matmul_id_slotted_page,
]
