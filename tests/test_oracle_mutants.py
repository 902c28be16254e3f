"""Each planted mistake in the oracle (built with -DORACLE_MUTANT=n) must fail at least
one pin; this shows the pins can tell a correct oracle from a plausibly wrong one."""
import numpy as np
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


# Planted mistakes in the flash-decoding merge (numpy part of the oracle): each must fail the
# split/merge pin.
def _merge_flipped_weights(m, l, a):
    mm = m.max(axis=0)
    w = np.where(np.isneginf(m), 0.0, np.exp(mm[None] - m))  # exp(m - m_i) instead of exp(m_i - m)
    ll = (w * l).sum(axis=0)
    aa = (w[..., None] * a).sum(axis=0)
    return mm, ll, aa, aa / ll[..., None], mm + np.log(ll)


def _merge_unweighted_l(m, l, a):
    mm = m.max(axis=0)
    w = np.where(np.isneginf(m), 0.0, np.exp(m - mm[None]))
    ll = l.sum(axis=0)  # l summed without the rescale
    aa = (w[..., None] * a).sum(axis=0)
    return mm, ll, aa, aa / ll[..., None], mm + np.log(ll)


def _merge_first_max(m, l, a):
    mm = np.where(np.isneginf(m[0]), m.max(axis=0), m[0])  # reference from the first chunk only
    w = np.where(np.isneginf(m), 0.0, np.exp(np.minimum(m - mm[None], 0.0)))
    ll = (w * l).sum(axis=0)
    aa = (w[..., None] * a).sum(axis=0)
    return mm, ll, aa, aa / ll[..., None], mm + np.log(ll)


@pytest.mark.parametrize("broken", [_merge_flipped_weights, _merge_unweighted_l, _merge_first_max],
                         ids=lambda f: f.__name__)
def test_merge_mutant_is_caught(broken, monkeypatch):
    monkeypatch.setattr(oracle, "merge_partials", broken)
    orc = oracle.Oracle(threads=2)
    with pytest.raises(AssertionError):
        oracle_pins.check_split_merge_equals_unsplit(orc)
