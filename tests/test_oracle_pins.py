"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""

import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle)


def test_three_pass_and_decode_bounds():
    """Oracle argument checks."""
    import numpy as np
    with pytest.raises(ValueError):
        oracle.group_size(-1, 4)
    with pytest.raises(ValueError):
        oracle.group_size(4, 0)
    assert oracle.group_size(0, 4) == 1
    k = np.zeros((1, 4, 1, 4))
    with pytest.raises(ValueError):
        oracle.bifocal_decode(np.zeros((1, 1, 4)), k, k, 5, 1, 2, 1e4)
