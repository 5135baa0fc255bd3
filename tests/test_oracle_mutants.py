"""Each deliberate mistake planted in a build of the oracle must fail at least one pin.

The mutants are compiled from the oracle's own source with -DKLA_ORACLE_MUTANT=n
(CPU only): 1 predict before forget, 2 eps outside the denominator, 3 sign of the
residual, 4 eta dropped, 5 read before write, 6 per-channel gate on the value
channels, 7 transposed read, 8 the raw-beta mode still taking the KLA step, 9 the query
scale dropped, 10 (backward) the step's dependence on ||k|| dropped, 11 (backward) the
residual's path back into the state dropped.
"""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11])
def test_mutant_is_caught(mutant):
    m = oracle.load(mutant)
    assert m.lib.kla_oracle_mutant_id() == mutant
    caught = []
    for pin in oracle_pins.PINS:
        try:
            pin(m)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
