"""Each planted mistake in the oracle (compiled with -DOQ4_MUTANT=n) must be
caught by at least one pin, which shows the pins can tell a wrong oracle from
the right one.  Mistakes: 1 ties-to-even codes, 2 ties-to-even zero, 3 high
nibble for the even index, 4 no widening of the range to 0, 5 scale divided by
16, 6 rounding after adding the zero, 7 zero from +lo, 8 factored dot without
the zero term, 9 dequant with q + zero, 10 transposed weight operand, 11 wrong
group index; symmetric scheme: 12 ties away from zero, 13 scale max|w|/8,
14 codes stored as q + 7; compact metadata: 15 binary16 by truncation, 16
zero nibbles swapped."""
import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = list(range(1, 17))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_mutant_is_caught(mutant, tmp_path):
    o = oracle.load_mutant(mutant, str(tmp_path))
    assert o.mutant == mutant
    caught = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
