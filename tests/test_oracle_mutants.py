"""Mutation test for the oracle's pins (CPU only).

Each mutant is a copy of the oracle built with one plausible mistake planted
(unbiased variance, eps outside the square root, a dropped or sign-flipped
term of dx, dgamma on raw x, a transposed channels_last index, gamma indexed
by group, statistics over one channel, parameter gradients over one sample).
The pins must reject every one of them.
"""
import pytest

import oracle
from tests import pins

MUTANTS = list(range(1, 11))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_every_mutant_fails_a_pin(mutant, tmp_path):
    o = oracle.Oracle(mutant, outdir=str(tmp_path))
    assert o.mutant == mutant
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
