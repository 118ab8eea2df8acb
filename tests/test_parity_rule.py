"""The list-acceptance rule of tests/parity.py on hand-built score vectors (CPU).

Each case builds scores whose oracle selection is known, then hands the rule
a list that differs from it in one specific way: a swap of pages tied with
the cutoff (accepted as a score tie), one page more or fewer where the
running mass crosses gamma within the mass tolerance (a mass tie), and the
ways a list can be wrong (a swap across a real score gap, a count off where
the mass is far from gamma, duplicates, out-of-range ids).
"""

import numpy as np
import pytest

import oracle.asp_oracle as O
from tests import parity


def _scores_with_mass(masses):
    """Scores whose page masses (softmax) are exactly proportional to `masses`."""
    return np.log(np.asarray(masses, dtype=np.float64))


def test_exact_list():
    s = _scores_with_mass([0.5, 0.3, 0.15, 0.05])
    assert parity.list_verdict([0, 1, 2], s, 0.9) == "exact"


def test_swap_of_pages_tied_with_the_cutoff_is_a_score_tie():
    # pages 2 and 3 tie within 1e-7 relative at the cutoff: either may be kept
    s = np.array([3.0, 2.0, 1.0, 1.0 - 1e-7, -5.0])
    want = O.coverage_select(s, 0.9)
    assert 2 in want and 3 not in want
    g = sorted(set(want.tolist()) - {2} | {3})
    assert parity.list_verdict(g, s, 0.9) == "score_tie"


def test_swap_across_a_real_gap_fails():
    s = np.array([3.0, 2.0, 1.0, 1.0 - 1e-3, -5.0])
    want = O.coverage_select(s, 0.9)
    g = sorted(set(want.tolist()) - {2} | {3})
    v = parity.list_verdict(g, s, 0.9)
    assert v not in parity.ACCEPTED


def test_tie_width_is_relative_to_the_cutoff_score():
    # a gap of 5e-6 is below 1e-6 of the largest |score| (10) but above 1e-6
    # of the cutoff score (~0.5): not a tie
    s = np.array([10.0, 0.5, 0.5 - 5e-6, -20.0])
    want = O.coverage_select(s, 0.9999)
    assert want.tolist() == [0, 1]
    assert parity.list_verdict([0, 2], s, 0.9999) not in parity.ACCEPTED
    # the same gap at a cutoff score of ~10 is a tie
    s2 = np.array([20.0, 10.0, 10.0 - 5e-6, -20.0])
    want2 = O.coverage_select(s2, 0.99993)
    assert want2.tolist() == [0, 1]
    assert parity.list_verdict([0, 2], s2, 0.99993) == "score_tie"


def test_one_page_more_at_the_gamma_crossing_is_a_mass_tie():
    # cumulative masses 0.6, 0.9 - 4e-7, ...: at gamma = 0.9 the oracle keeps
    # three pages, but two reach gamma within 1e-6, so keeping two, or keeping
    # three when the running mass is 4e-7 past gamma, are both mass ties
    m = np.array([0.6, 0.3 - 4e-7, 0.05, 0.05 + 4e-7])
    s = _scores_with_mass(m)
    want = O.coverage_select(s, 0.9)
    assert len(want) == 3
    assert parity.list_verdict([0, 1], s, 0.9) == "mass_tie"
    # one page more than the oracle where the crossing is that close
    m2 = np.array([0.6, 0.3 + 4e-7, 0.05, 0.05 - 4e-7])
    s2 = _scores_with_mass(m2)
    assert len(O.coverage_select(s2, 0.9)) == 2
    assert parity.list_verdict([0, 1, 2], s2, 0.9) == "mass_tie"


def test_count_off_where_the_mass_is_far_from_gamma_fails():
    m = np.array([0.6, 0.25, 0.1, 0.05])
    s = _scores_with_mass(m)
    assert len(O.coverage_select(s, 0.9)) == 3
    assert parity.list_verdict([0, 1], s, 0.9).startswith("mass")
    assert parity.list_verdict([0, 1, 2, 3], s, 0.9).startswith("not minimal")


def test_mass_tie_must_still_be_a_top_set():
    m = np.array([0.6, 0.3 - 4e-7, 0.05, 0.05 + 4e-7])
    s = _scores_with_mass(m)
    # two pages reaching gamma, but not the top two
    assert parity.list_verdict([0, 3], s, 0.9) not in parity.ACCEPTED


def test_budget_mode_and_gamma_one():
    s = np.array([3.0, 2.0, 1.0, 1.0, 0.0])
    assert parity.list_verdict([0, 1, 2], s, 0.5, budget=3) == "exact"
    assert parity.list_verdict([0, 1, 3], s, 0.5, budget=3) == "score_tie"
    assert parity.list_verdict([0, 1], s, 0.5, budget=3).startswith("budget count")
    assert parity.list_verdict([0, 1, 4], s, 0.5, budget=3) not in parity.ACCEPTED
    assert parity.list_verdict([0, 1, 2, 3, 4], s, 1.0) == "exact"
    assert parity.list_verdict([0, 1, 2, 3], s, 1.0).startswith("gamma=1")


def test_invalid_lists_fail():
    s = np.array([3.0, 2.0, 1.0])
    assert parity.list_verdict([0, 0], s, 0.9).startswith("invalid")
    assert parity.list_verdict([0, 5], s, 0.9).startswith("invalid")
    assert parity.list_verdict([], s, 0.9) == "empty list"


def test_gamma_is_taken_at_float32():
    # the ABI passes gamma as a float: 0.9 becomes 0.89999997615814208984375,
    # and the oracle's decision is taken at that value
    m = np.array([0.6, 0.3 - 1e-8, 0.1 + 1e-8])
    s = _scores_with_mass(m)
    assert parity.list_verdict([0, 1], s, 0.9) == "exact"


def test_tally_bounds_mass_ties():
    t = parity.VerdictCounts("unit")
    for _ in range(300):
        t.add("exact")
    t.add("mass_tie")
    t.finish()
    t.add("mass_tie")
    with pytest.raises(AssertionError):
        t.finish()
    with pytest.raises(AssertionError):
        t.add("not a top set")
