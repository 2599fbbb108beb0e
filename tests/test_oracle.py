"""The CPU oracle against its pins (no GPU)."""

import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def test_ulp16_definition():
    import numpy as np
    u = oracle.ulp16(np.array([0.0, 1.0, 1.999, 2.0, 65504.0, 2.0 ** -14, 2.0 ** -15, -3.0]))
    assert list(u) == [2.0 ** -24, 2.0 ** -10, 2.0 ** -10, 2.0 ** -9, 32.0, 2.0 ** -24,
                       2.0 ** -24, 2.0 ** -9]
