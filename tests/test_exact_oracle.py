"""The exact-mode oracle against its pins, and the pins against planted mistakes."""
import pytest

import pins_exact
from oracle.exact_mode import N_MUTANTS, ExactOracle


@pytest.mark.parametrize("pin", pins_exact.EXACT_PINS, ids=lambda p: p.__name__)
def test_exact_oracle_pin(oracle, pin):
    pin(ExactOracle(), oracle)


@pytest.mark.parametrize("mutant", range(1, N_MUTANTS + 1))
def test_exact_pins_catch_planted_mistake(mutant, oracle):
    m = ExactOracle(mutant=mutant)
    caught = []
    for pin in pins_exact.EXACT_PINS:
        try:
            pin(m, oracle)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught planted mistake {mutant} of the exact oracle"
