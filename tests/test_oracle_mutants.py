"""Each deliberately wrong oracle build must fail at least one pin.

The mistakes are planted in the oracle's C source behind ORC_MUTANT and built
on the CPU only: a dropped ReLU, a dropped key scale, keys read from the wrong
sequence, an off-by-one visibility count, the reverse tie rule, a window that
misses the query's own token, a dropped term of the dot product, keys used as
values, a flipped logit sign, ignored head weights, a dropped query scale, an
attention sink that also adds to the numerator, one left out of the
denominator, one multiplied by the softmax scale.
"""
import pytest

import oracle
import oracle_pins

MUTANTS = {1: "no ReLU", 2: "no k_scale", 3: "wrong sequence", 4: "visibility off by one",
           5: "reverse tie rule", 6: "window without self", 7: "dropped dot term",
           8: "K used as V", 9: "negated logits", 10: "weights ignored", 11: "no q_scale",
           19: "sink in the numerator", 20: "sink left out of the denominator",
           21: "sink scaled like a logit"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m].replace(" ", "_"))
def test_mutant_is_caught(mutant):
    path = oracle.mutant_build(mutant)
    oracle._lib(mutant, path)          # load the scratch build under this key
    oracle._LIBS[mutant] = oracle._LIBS[path]
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant=mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
