"""The oracle against its pins (no GPU): golden values from the pages, torch's
float8 and scaled-dot-product-attention routines, invariants and brute force."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL, ids=lambda f: f.__name__)
def test_oracle_pin(oracle, pin):
    pin(oracle)


def test_oracle_threads(oracle):
    assert oracle.threads() >= 1
