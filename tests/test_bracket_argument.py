"""The directed-rounding bracket of the fp64 cross-rank sum, in exact arithmetic.

The EP combine's fp64 forms sum the rank partials (float32 values) in rank
order twice in float32, every add rounded toward -inf (lo) and toward +inf
(hi), and take bf16(lo) as the result wherever bf16(lo) == bf16(hi).  The
claim it rests on: lo <= s <= hi for the binary64 sum s taken in the same
order from +0, so that, bf16 rounding being monotone, equal ends give the bf16
of s.  Checked here on random partial lists (mixed signs, spans of up to 200
binades, exact cancellations) with every rounding done exactly on rationals;
no GPU and no oracle code involved.  The kernel itself is checked against the
oracle bit for bit by the GPU parity tests."""
from __future__ import annotations

import math
import random
from fractions import Fraction

import numpy as np

from tests import exact

F32_MAX = Fraction(float(np.finfo(np.float32).max))


def _down(v: Fraction) -> Fraction | float:
    """Largest float32 <= v (as an exact value), or -inf."""
    r = exact.round_f32(v)
    if math.isinf(r):
        return F32_MAX if r > 0 else -math.inf
    if Fraction(r) > v:
        r = float(np.nextafter(np.float32(r), np.float32(-np.inf)))
        if math.isinf(r):
            return -math.inf
    return Fraction(r)


def _up(v: Fraction) -> Fraction | float:
    """Smallest float32 >= v, or +inf."""
    r = exact.round_f32(v)
    if math.isinf(r):
        return math.inf if r > 0 else -F32_MAX
    if Fraction(r) < v:
        r = float(np.nextafter(np.float32(r), np.float32(np.inf)))
        if math.isinf(r):
            return math.inf
    return Fraction(r)


def _f64(v: Fraction) -> Fraction:
    s, m = exact.round_binary(v, 53, -1022, 1023)
    assert m != math.inf
    return s * m


def _partials(rng: random.Random, n: int, span: int) -> list[Fraction]:
    base = rng.randint(-60, 40)
    out = []
    for _ in range(n):
        e = base + rng.randint(0, span)
        m = rng.randint(1 << 23, (1 << 24) - 1)
        out.append(Fraction(rng.choice((-1, 1)) * m) * Fraction(2) ** (e - 23))
    if rng.random() < 0.2 and n >= 2:             # an exact cancellation
        out[1] = -out[0]
    return out


def _bracket(parts):
    lo = hi = Fraction(0)
    for p in parts:
        lo = _down(lo + p) if not isinstance(lo, float) else lo
        hi = _up(hi + p) if not isinstance(hi, float) else hi
    return lo, hi


def _bf16(v) -> int:
    if isinstance(v, float):                     # +-inf
        return 0xFF80 if v < 0 else 0x7F80
    return 0 if v == 0 else exact.round_bf16_bits(v)


def test_bracket_holds_the_binary64_sum_and_decides_its_bf16():
    rng = random.Random(20261202)
    decided = 0
    cases = 3000
    for i in range(cases):
        n = rng.randint(1, 8)
        parts = _partials(rng, n, rng.choice((2, 8, 30, 60, 200)))
        s = Fraction(0)
        for p in parts:
            s = _f64(s + p)
        lo, hi = _bracket(parts)
        assert (lo if not isinstance(lo, float) else -math.inf) <= s
        assert s <= (hi if not isinstance(hi, float) else math.inf)
        if _bf16(lo) == _bf16(hi):
            decided += 1
            assert _bf16(lo) == _bf16(s), (i, parts)
    # most elements are decided by the bracket alone
    assert decided > cases * 0.6


def test_ties_and_cancellations():
    """Partials 1 + 2^-8 sit exactly on a bf16 midpoint: a third partial below
    an fp32 ulp of the sum leaves the bracket undecided whenever s lies
    beyond the tie, and the ends then round apart; an exact cancellation is
    the same value at both ends (the rounded-down end's -0 is not modelled
    here: a zero counts as +0 on both sides)."""
    one, q = Fraction(1), Fraction(1, 256)
    for third, decided in ((Fraction(1, 2**30), False), (Fraction(-1, 2**30), True),
                           (Fraction(1, 2**12), True), (Fraction(0), True)):
        lo, hi = _bracket([one, q, third])
        assert (_bf16(lo) == _bf16(hi)) == decided, third
    lo, hi = _bracket([one, -one])
    assert lo == hi == 0
