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
