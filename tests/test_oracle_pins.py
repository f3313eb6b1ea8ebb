"""The oracle against its pins, and planted mistakes against the pins (CPU only)."""
import pytest

from oracle import build as obuild
from oracle.oracle import Oracle
from tests import oracle_pins as P

MUTANTS = list(range(1, 34))


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    assert oracle.mutant() == 0
    pin(oracle)


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistake_is_caught(tmp_path, mutant):
    """Each planted mistake in the oracle fails at least one pin."""
    o = Oracle(path=obuild.build(mutant=mutant, openmp=False, out_dir=str(tmp_path)))
    assert o.mutant() == mutant
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"
