"""The fp64 oracle against its pins (closed forms, library special cases,
finite differences, invariants and the pages' tiled algorithm)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np
    with pytest.raises(ValueError):
        orc.online_softmax_stats(np.zeros(3), 0)
