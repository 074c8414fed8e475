"""Pins for the oracle's E2M1 / E4M3 formats against the format definitions.

Nothing here compares the oracle with itself: expected values come from the
hand-worked fixtures under tests/golden/ (each cites the format definition it
follows), from invariants every correct rounding has (round trip, monotonicity,
ties to even at every midpoint, saturation), and from brute force over the grid
with exact rational arithmetic.
"""

from fractions import Fraction

import numpy as np
import pytest

from conftest import golden_lines


def _f32(x):
    return np.float32(float(x))


def test_e2m1_decode_matches_format_table(orc):
    rows = golden_lines("e2m1_values.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code = int(code_s, 16)
        v = orc.e2m1_decode(code)
        assert v == float(val_s)
        assert np.signbit(v) == val_s.startswith("-")


def test_e2m1_roundtrip_every_code(orc):
    vals = np.array([orc.e2m1_decode(c) for c in range(16)], np.float32)
    assert list(orc.e2m1_rne(vals)) == list(range(16))


def test_e2m1_ties_and_saturation(orc):
    rows = golden_lines("e2m1_ties.txt")
    q = np.array([_f32(a) for a, _ in rows], np.float32)
    want = [int(b, 16) for _, b in rows]
    assert list(orc.e2m1_rne(q)) == want


def test_e2m1_nearest_bruteforce(orc):
    """Every code is a nearest grid point (exact rationals), ties to even mantissa."""
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2),
            Fraction(3), Fraction(4), Fraction(6)]
    rng = np.random.default_rng(1)
    q = np.concatenate([
        rng.uniform(-8, 8, 4000).astype(np.float32),
        # values within a few ulps of every midpoint
        np.array([np.nextafter(np.float32(m), np.float32(s * 10), dtype=np.float32)
                  for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0) for s in (-1, 1)], np.float32),
    ])
    codes = orc.e2m1_rne(q)
    for x, c in zip(q, codes):
        mag = abs(Fraction(float(x)))
        d = [abs(g - mag) for g in grid]
        best = min(d)
        winners = [i for i, di in enumerate(d) if di == best]
        want = winners[0] if len(winners) == 1 else [w for w in winners if w % 2 == 0][0]
        assert (c & 7) == want, (x, c)
        assert (c >> 3) == int(np.signbit(x))


def test_e2m1_monotone(orc):
    q = np.sort(np.random.default_rng(2).uniform(0, 10, 20000).astype(np.float32))
    mags = orc.e2m1_rne(q) & 7
    assert np.all(np.diff(mags.astype(int)) >= 0)


def test_e2m1_product_table(orc):
    """All 16 x 16 code products are exact multiples of 1/4 with |p| <= 36."""
    seen = set()
    for a in range(16):
        for b in range(16):
            p = orc.e2m1_decode(a) * orc.e2m1_decode(b)
            exact = Fraction(orc.e2m1_decode(a)) * Fraction(orc.e2m1_decode(b))
            assert Fraction(p) == exact
            assert (exact * 4).denominator == 1 and abs(exact) <= 36
            seen.add(exact)
    mags = {Fraction(x) for x in (0, 0.5, 1, 1.5, 2, 3, 4, 6)}
    assert seen == {s * a * b for a in mags for b in mags for s in (1, -1)}


def test_e4m3_decode_points(orc):
    for code_s, val_s in golden_lines("e4m3_values.txt"):
        assert orc.e4m3_decode(int(code_s, 16)) == float(val_s)
    assert np.isnan(orc.e4m3_decode(0x7F)) and np.isnan(orc.e4m3_decode(0xFF))
    assert orc.e4m3_decode(0xB8) == -1.0


def test_e4m3_roundtrip_every_finite_code(orc):
    vals = np.array([orc.e4m3_decode(c) for c in range(127)], np.float32)
    assert list(orc.e4m3_rne(vals)) == list(range(127))
    # value order equals code order, subnormal spacing 2^-9
    assert np.all(np.diff(vals.astype(np.float64)) > 0)
    assert all(vals[c] == c * 2.0 ** -9 for c in range(8))


def test_e4m3_ties_and_saturation(orc):
    rows = golden_lines("e4m3_ties.txt")
    v = np.array([_f32(a) for a, _ in rows], np.float32)
    assert list(orc.e4m3_rne(v)) == [int(b, 16) for _, b in rows]


def test_e4m3_every_midpoint_ties_to_even(orc):
    vals = [Fraction(orc.e4m3_decode(c)) for c in range(127)]
    mids, want = [], []
    for c in range(126):
        m = (vals[c] + vals[c + 1]) / 2
        assert Fraction(float(np.float32(float(m)))) == m  # midpoints are fp32-exact
        mids.append(float(m))
        want.append(c if c % 2 == 0 else c + 1)
        # one ulp either side goes to the nearer code
        lo = np.nextafter(np.float32(float(m)), np.float32(0), dtype=np.float32)
        hi = np.nextafter(np.float32(float(m)), np.float32(1e9), dtype=np.float32)
        assert orc.e4m3_rne(np.array([lo], np.float32))[0] == c
        assert orc.e4m3_rne(np.array([hi], np.float32))[0] == c + 1
    assert list(orc.e4m3_rne(np.array(mids, np.float32))) == want
