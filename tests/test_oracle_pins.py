"""The CPU oracle against its pins, and the pins against planted mistakes."""
import os
import tempfile

import numpy as np
import pytest

import pins
from oracle import oracle as oracle_mod

N_MUTANTS = 11


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle, pin):
    pin(oracle)


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory(prefix="oracle_mutants_") as d:
        yield d


@pytest.mark.parametrize("mutant", range(1, N_MUTANTS + 1))
def test_pins_catch_planted_mistake(mutant, mutant_dir):
    path = oracle_mod.build(out=os.path.join(mutant_dir, f"mutant{mutant}.so"), mutant=mutant, force=True)
    m = oracle_mod.Oracle.load(path)
    assert m.mutant == mutant
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(m)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught planted mistake {mutant}"


def test_thread_count_never_changes_bits():
    from deterministic_arithmetic_gb300 import synthetic as S

    d = S.tiny().generate(1)
    one = oracle_mod.Oracle.load(threads=1)
    many = oracle_mod.Oracle.load(threads=7)
    a = one.fwd(d["x"], d["a"], d["b"], 2.0)
    b = many.fwd(d["x"], d["a"], d["b"], 2.0)
    assert np.array_equal(a["u"], b["u"]) and np.array_equal(a["delta_y"].view(np.uint32), b["delta_y"].view(np.uint32))
    ga = one.bwd(d["dy"], d["x"], d["a"], d["b"], a["u"], 2.0)
    gb = many.bwd(d["dy"], d["x"], d["a"], d["b"], b["u"], 2.0)
    for k in ga:
        assert np.array_equal(ga[k].view(np.uint8), gb[k].view(np.uint8)), k
