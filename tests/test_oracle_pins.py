"""The oracle against its pins (CPU only)."""

import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(o, pin):
    pin(o)


def test_threaded_matmul_matches_single_thread(o):
    import q2k_workloads as wl
    x, w = wl.make_matmul_inputs(5, 3, 37, 512)
    y1, s1 = o.matmul(x, w, 37, threads=1)
    y4, s4 = o.matmul(x, w, 37, threads=4)
    assert (y1 == y4).all() and (s1 == s4).all()


def test_rejects_bad_shapes(o):
    import numpy as np
    with pytest.raises(oracle.OracleError):
        o.matmul(np.zeros((1, 200), np.float32), np.zeros(84, np.uint8), 1)
    with pytest.raises(oracle.OracleError):
        o.gather(np.zeros(84, np.uint8), 1, 200, [0])


def test_matmul_rows_is_matmul_restricted_to_those_rows(o):
    """oracle.matmul_rows (the sampled-row helper) picks the right weight rows:
    its columns equal the full product's columns, bit for bit, for any row set
    (unordered, repeated, first and last rows)."""
    import numpy as np
    import q2k_workloads as wl
    n, k = 29, 768
    x, w = wl.make_matmul_inputs(31, 3, n, k)
    y, s = o.matmul(x, w, n, threads=2)
    for rows in ([0], [n - 1], [5, 2, 17], [3, 3, 28, 0], list(range(n))):
        yr, sr = oracle.matmul_rows(x, w, n, rows, threads=2)
        assert np.array_equal(yr, y[:, rows]) and np.array_equal(sr, s[:, rows])
