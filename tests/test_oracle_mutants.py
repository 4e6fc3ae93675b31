"""Every planted mistake in the oracle must trip at least one pin (CPU only).

The mistakes are compiled into separate builds of the oracle source with
ORACLE_MUTANT=n: (1) causal bound off by one, (2) wrong GQA head map, (3)
block table ignored, (4) scale dropped, (5) K and V swapped, (6) a term
dropped from the softmax denominator, (7) causal offset with its sign flipped,
(8) the K/V append writing one slot too far, (9) an explicit mask subtracted
instead of added, (10) a ragged batch's causal offset taken from the longest
query instead of the sequence's own, (11) the softmax's max not subtracted
(exact in real arithmetic, overflows on large scores), (12) the slot off by
one within its page, (13) the last key of every context dropped.  Each keeps
every index in bounds, so a mutant fails a pin instead of crashing the run.
"""
import pytest

import oracle
import pins

MUTANTS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistake_is_caught(mutant):
    lib = oracle.load(mutant)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
