"""The parity tolerance check itself (no GPU): an output the kernel never
wrote (left as NaN by the tests' prefill) or an infinity must fail it."""
import numpy as np
import pytest

from _harness import check_close


def test_check_close_accepts_within_tolerance():
    want = np.array([1.0, -2.0, 0.0])
    mag = np.array([1.0, 2.0, 0.5])
    assert check_close("x", want + 0.5e-5 * mag, want, mag) <= 0.5e-5 + 1e-12


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf, 1e-3])
def test_check_close_rejects_nan_inf_and_large_errors(bad):
    want = np.zeros(4)
    mag = np.ones(4)
    got = want.copy()
    got[2] = bad
    with pytest.raises(AssertionError):
        check_close("x", got, want, mag)
