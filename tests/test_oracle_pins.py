"""The oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(orc, pin):
    pin(orc)


def test_no_visible_key_is_reported(orc):
    import numpy as np
    Q = np.ones((1, 1, 2, 4))
    K = np.ones((1, 1, 3, 4))
    out = orc.sdpa(Q, K, K, mask_kind=oracle.MASK_KEY_PADDING,
                   key_lengths=np.array([0], np.int32))
    assert orc.last_bad_rows == 2 and np.all(np.isnan(out))
