"""The oracle against its pins (CPU only)."""
import pytest

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    o = oracle.load()
    assert o.mutant == 0
    pin(o)


def test_oracle_config1_bound_full():
    """The page's bound on every row of the full 4096 x 4096 xorshift matrix."""
    from oracle_pins import pin_matrix_bound
    pin_matrix_bound(oracle.load(), N=4096, K=4096)
