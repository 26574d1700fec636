"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle_pins import PINS, pin_hand_example, _small


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_recurrence_pin(pin):
    pin(oracle.recurrence)


@pytest.mark.parametrize("form", [oracle.quadratic, oracle.assoc_scan], ids=["quadratic", "assoc_scan"])
def test_other_forms_hand_example(form):
    pin_hand_example(lambda x, dt, A, B, C, D, init: form(x, dt, A, B, C, D, init))


def test_row_subset_and_threads_agree():
    inp = _small(21, b=2, L=33, H=4, P=5, N=6, G=2)
    y, f = oracle.recurrence(**inp, nthreads=1)
    y8, f8 = oracle.recurrence(**inp, nthreads=8)
    assert np.array_equal(y, y8) and np.array_equal(f, f8)
    b, L, H, P = y.shape
    rows = [0, 7, 19, b * H * P - 1]
    yr, fr = oracle.recurrence(**inp, rows=rows, nthreads=3)
    for i, r in enumerate(rows):
        bb, h, p = r // (H * P), (r // P) % H, r % P
        assert np.array_equal(yr[i], y[bb, :, h, p])
        assert np.array_equal(fr[i], f[bb, h, p])


def test_rejects_bad_arguments():
    inp = _small(22)
    with pytest.raises(ValueError):
        oracle.recurrence(inp["x"][:, :, :3], inp["dt"], inp["A"], inp["B"], inp["C"])
    with pytest.raises(RuntimeError):
        oracle.recurrence(**inp, rows=[10 ** 9])
