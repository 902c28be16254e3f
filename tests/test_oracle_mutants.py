"""Each planted mistake in the oracle (built with -DORACLE_MUTANT=n) must fail at least
one pin; this shows the pins can tell a correct oracle from a plausibly wrong one."""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    1: "scale dropped from the scores",
    2: "one term dropped from the softmax denominator",
    3: "causal mask lets one future key through",
    4: "score operands transposed",
    5: "row max dropped from the LSE",
    6: "scale dropped from dQ",
    7: "wrong operand in dK",
    8: "D computed without the P weights",
    9: "P not transposed in dV",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"m{m}")
def test_mutant_is_caught(mutant):
    orc = oracle.Oracle(mutant=mutant, threads=2)
    assert orc.lib.fa_oracle_mutant_id() == mutant
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
            break
    assert failed, f"no pin caught mutant {mutant}: {MUTANTS[mutant]}"
