"""The tolerance check itself rejects what it should."""
import numpy as np
import pytest

from tests.parity import assert_close


def test_accepts_within_bar():
    ref = np.array([0.0, 0.1, 1.0, -3.0])
    assert_close(ref + np.array([1.9e-3, -1.9e-3, 1.9e-3, 1.9e-3]), ref)


@pytest.mark.parametrize("delta,idx", [(2.1e-3, 0), (2.1e-3, 2), (np.nan, 1)])
def test_rejects_outside_bar(delta, idx):
    ref = np.array([0.0, 0.1, 1.0, -3.0])
    bad = ref.copy()
    bad[idx] += delta
    with pytest.raises(AssertionError):
        assert_close(bad, ref)
