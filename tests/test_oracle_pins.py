"""The CPU oracle against its pins (closed forms, library routines, brute
force, hand-worked fixtures and chi-square losslessness).  CPU only."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc.load())
