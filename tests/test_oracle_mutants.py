"""Each planted mistake in the oracle (a flipped sign, the decay applied to
the write term, a dropped write term, a transposed read-out, the write vector
taken after the step, the tree read as a chain, the accepted path replayed
backwards) must fail at least one pin.  The mistakes are compiled into
throw-away copies of the oracle on the CPU; the real oracle is untouched."""

import os

import pytest

import oracle
from tests import pins

MUTANTS = ["ORC_MUTANT_SIGN", "ORC_MUTANT_DECAY_ON_WRITE", "ORC_MUTANT_DROP_WRITE",
           "ORC_MUTANT_TRANSPOSE", "ORC_MUTANT_U_AFTER_STEP", "ORC_MUTANT_IGNORE_TREE",
           "ORC_MUTANT_REVERSED_PATH"]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistake_is_caught(tmp_path, mutant):
    so = oracle.compile_library(os.path.join(tmp_path, f"{mutant}.so"), (mutant,))
    lib = oracle.load(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            err = pin(lib)
        except Exception:
            err = float("inf")
        if not err <= pins.PIN_TOL:
            caught.append(pin.__name__)
    assert caught, f"{mutant} passed every pin"
