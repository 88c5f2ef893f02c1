"""The oracle against its pins: worked examples, brute force, library special
cases and the identities the pages state (see ``oracle_pins``)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(None)
