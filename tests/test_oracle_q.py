"""Pins of the oracle's fill count q against what the pages and the algebra fix."""
import json
import os
import random
from fractions import Fraction

import pytest

from oracle.control import fill_count, round_half_away, round_half_away_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q_page_examples.json")


def test_page_examples():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        S = 10_000
        h = c.get("hits", 0)
        fc = fill_count(c["m"], h, S, c["B_P"], c["B_H"])
        assert fc.q == c["q"], c["cite"]
        if "cpu" in c:
            assert c["m"] - fc.q == c["cpu"], c["cite"]


def test_closed_form_balances_the_two_branches():
    """q* = m*B_P/B_H is exactly where q*S/B_P equals (m-q*)S/(B_H-B_P)
    (explainer section 5); checked in exact rationals, independent of the
    oracle's float64 path."""
    rng = random.Random(1)
    for _ in range(500):
        m = rng.randint(1, 300)
        BP = Fraction(rng.randint(1, 1000), rng.randint(1, 50))
        BH = BP + Fraction(rng.randint(1, 1000), rng.randint(1, 50))
        S = Fraction(rng.randint(1, 10**7))
        q = m * BP / BH
        assert q * S / BP == (m - q) * S / (BH - BP)
        # and no other split balances them: the branch times move in opposite directions
        assert (q + Fraction(1, 7)) * S / BP > (m - q - Fraction(1, 7)) * S / (BH - BP)


def test_float_path_agrees_with_exact_rationals():
    rng = random.Random(2)
    pairs = [(25.0, 75.0), (52.7, 120.0), (25.0, 90.0), (52.7, 150.0), (11.8, 47.5), (49.0, 53.8),
             (52.7, 77.3), (25.1, 63.2), (25.3, 56.7), (51.5, 178.0)]
    for BP, BH in pairs:
        for m in range(0, 257):
            fc = fill_count(m, 0, 10**6, BP, BH)
            assert fc.q0 == fc.q0_exact, (m, BP, BH)
    for _ in range(2000):
        BP = round(rng.uniform(1, 100), 1)
        BH = round(BP + rng.uniform(0, 200), 1)
        m = rng.randint(1, 256)
        fc = fill_count(m, 0, 10**6, BP, BH)
        x = Fraction(m) * Fraction(str(BP)) / Fraction(str(BH))
        # a disagreement is only possible within one ulp of a half
        if fc.q0 != fc.q0_exact:
            assert abs(x - (Fraction(fc.q0_exact) - Fraction(1, 2))) < Fraction(1, 10**12)


def test_rounding_half_away_from_zero_on_exact_ties():
    # B_P/B_H = 25/90 = 5/18: m = 9 gives 2.5 exactly, and every 18 after it
    for m, q in [(9, 3), (27, 8), (45, 13), (63, 18), (81, 23), (99, 28), (117, 33)]:
        assert Fraction(m * 25, 90).denominator == 2
        assert fill_count(m, 0, 10**6, 25.0, 90.0).q == q
    assert round_half_away(0.5) == 1 and round_half_away(1.5) == 2 and round_half_away(2.5) == 3
    assert round_half_away(0.49999999999999994) == 0
    assert round_half_away_exact(Fraction(5, 2)) == 3


def test_at_least_one_fill_and_capacity_clamp():
    for m in range(1, 50):
        assert fill_count(m, 0, 1000, 0.001, 1000.0).q == 1          # ratio ~0 still fills one
        assert fill_count(m, 0, 1000, 77.0, 77.0).q == m              # B_H == B_P: fill every miss
        fc = fill_count(m, 5, 7, 77.0, 77.0)                          # only S - h = 2 free slots
        assert fc.q1 == m and fc.q == min(m, 2)
        assert fill_count(m, 4, 4, 77.0, 77.0).q == 0                 # every slot holds a hit
    assert fill_count(0, 3, 10, 1.0, 2.0).q == 0


def test_monotone_in_m_and_ratio():
    for BP, BH in [(52.7, 120.0), (25.0, 90.0), (1.0, 3.0)]:
        qs = [fill_count(m, 0, 10**6, BP, BH).q for m in range(1, 200)]
        assert all(a <= b for a, b in zip(qs, qs[1:]))
        assert all(b - a <= 1 for a, b in zip(qs, qs[1:]))
    for m in [1, 7, 33]:
        qs = [fill_count(m, 0, 10**6, r, 100.0).q for r in range(1, 101)]
        assert all(a <= b for a, b in zip(qs, qs[1:]))
