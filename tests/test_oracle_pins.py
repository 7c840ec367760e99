"""The CPU oracle against facts the mathematics fixes (see oracle_pins.py)."""
import numpy as np
import pytest

import oracle
from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.default())


def test_ulp_and_tolerance():
    # bf16 keeps 8 significant bits: ulp(v) = 2^(floor(log2 v) - 7)
    v = np.array([1.0, 1.99, 2.0, 0.75, 7232.0, 0.0, 2.0 ** -127, -3.0])
    want = np.array([2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -8, 32.0, 2.0 ** -133,
                     2.0 ** -133, 2.0 ** -6])
    assert np.array_equal(oracle.ulp_bf16(v), want)
    assert np.array_equal(oracle.tolerance(np.array([1.0])), np.array([4 * 2.0 ** -7 + 1e-3]))


def test_compare_flags_nan_and_excess():
    ref = np.array([1.0, 2.0, -0.5])
    assert oracle.compare(ref.copy(), ref)["ok"]
    bad = ref.copy()
    bad[1] = np.nan
    r = oracle.compare(bad, ref)
    assert not r["ok"] and r["n_bad"] == 1
    off = ref.copy()
    off[0] += 4 * 2.0 ** -7 + 1.01e-3
    assert not oracle.compare(off, ref)["ok"]
    off[0] = ref[0] + 4 * 2.0 ** -7 + 0.99e-3
    assert oracle.compare(off, ref)["ok"]


def test_oracle_rejects_bad_shapes():
    x = np.zeros((2, 8), dtype=np.uint16)
    w = np.zeros((3, 9), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm(x, w)
    with pytest.raises(TypeError):
        oracle.gemm(x.astype(np.float32), w)
