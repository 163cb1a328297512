"""The CPU oracle against its pins (no GPU needed)."""
import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())


def test_oracle_rejects_bad_arguments():
    o = oracle.default()
    with pytest.raises(ValueError):
        o.gemm_f64(np.ones((2, 3), np.float32), np.ones((4, 2), np.float32))
    with pytest.raises(TypeError):
        o.gemm_f64(np.ones((2, 3), np.float64), np.ones((3, 2), np.float32))
    with pytest.raises(RuntimeError):
        o.gemm_rows_f64(np.ones((2, 3), np.float32), np.ones((3, 2), np.float32), [2])
    with pytest.raises(RuntimeError):
        o.gemm_entries_f64(np.ones((2, 3), np.float32), np.ones((3, 2), np.float32), [0], [-1])
