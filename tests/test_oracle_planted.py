"""Each planted mistake in the oracle must make at least one pin fail.

The oracle source carries switches (-DORC_PLANT=n) that inject one plausible error each:
1 rotation sign, 2 window one token too wide, 3 interleaved GQA groups, 4 scale dropped,
5 wrong frequency exponent, 6 YaRN interpolation reversed, 7 ring index off by one,
8 RMSNorm over the sum of squares instead of their mean, 9 values of a shared K/V
projection normalised with the key gain instead of none.
The default build plants nothing (checked here too).
"""
import pytest

import oracle
import oracle_checks

PLANTS = [1, 2, 3, 4, 5, 6, 7, 8, 9]


def _failures(orc):
    failed = []
    for check in oracle_checks.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    return failed


def test_default_build_plants_nothing():
    assert oracle.default().lib.orc_plant() == 0


@pytest.mark.parametrize("plant", PLANTS)
def test_planted_mistake_is_caught(plant):
    orc = oracle.Oracle(plant)
    assert orc.lib.orc_plant() == plant
    failed = _failures(orc)
    assert failed, f"planted mistake {plant} passed every pin"
