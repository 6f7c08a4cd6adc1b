"""The CPU oracle against its pins (no GPU): hand-packed groups with
closed-form outputs, exact rational brute force, the pages' published byte
totals, bf16 rounding and glue closed forms."""
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)
