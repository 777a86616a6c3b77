"""The exact re-decision's double-single arithmetic against its stated error bounds (CPU).

The fix-up decides a flagged pair from q = 2 -/+ 2 a.b, where a.b is summed in double-single from
the fp32 vectors (hi) and the fp32 roundings of what they leave of the fp64 vectors (lo): fp32
products, their exact fma remainders, the cross terms and TwoSums (ds_dot and ds_chord_from_dot in
acf_kernels.cuh). Its comments bound the error of a.b against the dot product of the fp64 vectors by
30 2^-48 = 1.07e-13, and that of q by 2 x that + 2.2e-14; the decision window of 4e-13 adds the
tables' and the side test's own roundings. A decision is only as exact as these bounds.

Here the same sequence of operations is replayed with every fp32 operation rounded correctly from
its exact rational result (round to nearest, ties to even; an fma rounds once), on random unit
vectors and on the hard cases: nearly parallel and nearly antiparallel pairs, perpendicular pairs,
components near zero, coordinate axes. The exact dot product of the fp64 vectors is computed in
rational arithmetic. The test also checks that the bound is not vacuous: the worst error seen (7.1e-15
on these cases, mostly the fp64 vectors' own representation in hi + lo) is a noticeable fraction of
it.
"""
import math
import random
from fractions import Fraction

import numpy as np

DOT_ERR = 1.07e-13          # kDotErr in acf_kernels.cuh
CHORD_ERR = 2 * DOT_ERR + 2.2e-14


def f32(x: Fraction) -> Fraction:
    """x rounded to the nearest fp32 value (ties to even), as an exact rational. No overflow or
    subnormals arise here (|x| <= 4, and nonzero values far above 2^-126)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = -x if x < 0 else x
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix e so that 2^e <= a < 2^(e+1)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    scale = Fraction(2) ** (23 - e)          # a * scale in [2^23, 2^24)
    m = a * scale
    q, r = divmod(m.numerator, m.denominator)
    rem = Fraction(r, m.denominator)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
        q += 1
    return sign * Fraction(q) / scale


def add(a, b):
    return f32(a + b)


def sub(a, b):
    return f32(a - b)


def mul(a, b):
    return f32(a * b)


def fma(a, b, c):
    return f32(a * b + c)


def two_sum(a, b):
    s = add(a, b)
    bv = sub(s, a)
    av = sub(s, bv)
    t = add(sub(a, av), sub(b, bv))
    return s, t


def split(x: float):
    """The fp32 vector component and the fp32 rounding of what remains (as in vectors_kernel)."""
    hi = float(np.float32(x))
    lo = float(np.float32(x - hi))  # x - hi is exact in fp64
    return Fraction(hi), Fraction(lo)


def ds_dot(a, b):
    """The fix-up's double-single dot product of fp64 unit vectors a, b (returns dh, dl)."""
    ah, al = zip(*(split(v) for v in a))
    bh, bl = zip(*(split(v) for v in b))
    p = []
    r = Fraction(0)
    for c in range(3):
        pc = mul(ah[c], bh[c])
        e = fma(ah[c], bh[c], -pc)
        assert e == ah[c] * bh[c] - pc  # the remainder of a product is exact
        e = fma(ah[c], bl[c], e)
        e = fma(al[c], bh[c], e)
        e = fma(al[c], bl[c], e)
        r = e if c == 0 else add(r, e)
        p.append(pc)
    s1, t1 = two_sum(p[0], p[1])
    s2, t2 = two_sum(s1, p[2])
    return two_sum(s2, add(r, add(t1, t2)))


def chord_from_dot(dh, dl, sg):
    """q = 2 + 2 sg a.b as qh + ql (ds_chord_from_dot)."""
    qh, t = two_sum(Fraction(2), 2 * sg * dh)  # 2 sg dh is exact
    return qh, add(t, 2 * sg * dl)


def unit(v):
    v = np.asarray(v, dtype=np.float64)
    return v / np.linalg.norm(v)


def cases():
    rnd = random.Random(12345)
    out = []
    for _ in range(300):  # random directions
        out.append((unit([rnd.gauss(0, 1) for _ in range(3)]), unit([rnd.gauss(0, 1) for _ in range(3)])))
    for scale in (1e-2, 1e-4, 1e-6, 1e-8):  # nearly parallel and nearly antiparallel
        for _ in range(60):
            a = unit([rnd.gauss(0, 1) for _ in range(3)])
            d = unit([rnd.gauss(0, 1) for _ in range(3)]) * scale
            out.append((a, unit(a + d)))
            out.append((a, unit(-a + d)))
    for _ in range(120):  # nearly perpendicular
        a = unit([rnd.gauss(0, 1) for _ in range(3)])
        b = unit(np.cross(a, [rnd.gauss(0, 1) for _ in range(3)]) + a * rnd.uniform(-1e-3, 1e-3))
        out.append((a, b))
    for _ in range(120):  # components near zero (galaxies near the coordinate planes and poles)
        a = unit([rnd.uniform(-1e-7, 1e-7), rnd.gauss(0, 1), rnd.gauss(0, 1)])
        b = unit([rnd.gauss(0, 1), rnd.uniform(-1e-7, 1e-7), rnd.choice([-1, 1]) * rnd.uniform(0.5, 1)])
        out.append((a, b))
    for a in np.eye(3):  # axes
        for b in np.eye(3):
            out.append((a, b))
            out.append((a, -b))
    return out


def test_ds_dot_within_its_bound():
    worst = 0.0
    for a, b in cases():
        dh, dl = ds_dot(a, b)
        exact = sum(Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b))
        err = abs(float(dh + dl - exact))
        assert err <= DOT_ERR, (a, b, err)
        assert abs(dl) <= abs(dh) * 2.0 ** -23 + Fraction(1, 2 ** 149)  # normalised: dh is the fp32 rounding
        worst = max(worst, err)
    # the bound is not vacuous: the adversarial cases reach a noticeable part of it
    assert worst > DOT_ERR / 100, worst


def test_chord_from_dot_within_its_bound():
    for a, b in cases():
        dh, dl = ds_dot(a, b)
        for sg in (-1, 1):
            qh, ql = chord_from_dot(dh, dl, sg)
            a_f = [Fraction(float(x)) for x in a]
            b_f = [Fraction(float(x)) for x in b]
            exact = sum((x + sg * y) ** 2 for x, y in zip(a_f, b_f))  # |a + sg b|^2 of the fp64 vectors
            # (|a|^2 + |b|^2 of fp64 unit vectors is 2 within 1e-15)
            assert abs(float(qh + ql - exact)) <= CHORD_ERR + 1e-15, (a, b, sg)
