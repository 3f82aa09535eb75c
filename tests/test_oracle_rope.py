"""Pins for the oracle's RoPE table and rotation (CPU only).

Checked against: Python's libm (math.cos / math.sin, one value at a time),
the rotary definition's closed forms (position 0 is the identity, a unit
vector on the first axis lands on (cos, sin), pair norms are preserved, the
inner product of two rotated vectors depends only on the position difference),
and the proportional-RoPE denominator of the global layers.
"""

import math
from fractions import Fraction

import numpy as np

from oracle import rope


def _ulp32(a):
    return np.spacing(np.abs(a).astype(np.float32))


def test_table_matches_libm():
    for theta, R, D in [(1e4, 256, 256), (1e6, 128, 512)]:
        tab = rope.rope_table(theta, R, D, 140000)
        g = np.random.Generator(np.random.PCG64(11))
        for p, i in zip(g.integers(0, 140000, 4000), g.integers(0, R // 2, 4000)):
            ang = float(p) * theta ** (-2.0 * float(i) / D)
            c, s = np.float32(math.cos(ang)), np.float32(math.sin(ang))
            assert abs(tab[p, i, 0] - c) <= _ulp32(c) and abs(tab[p, i, 1] - s) <= _ulp32(s)


def test_position_zero_is_identity():
    tab = rope.rope_table(1e6, 128, 512, 4)
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1] == 0.0)
    x = np.random.Generator(np.random.PCG64(1)).normal(size=(5, 128)).astype(np.float32)
    assert np.array_equal(rope.rotate_half_f32(x, np.broadcast_to(tab[0], (5, 64, 2))), x)


def test_proportional_denominator():
    # global: only 128 of 512 dims rotate, frequencies over the full 512 dims
    tab = rope.rope_table(1e6, 128, 512, 2)
    for i in [1, 5, 63]:
        assert tab[1, i, 1] == np.float32(math.sin(1e6 ** (-2.0 * i / 512)))
        assert tab[1, i, 1] != np.float32(math.sin(1e6 ** (-2.0 * i / 128)))
    # local: all 256 dims, denominator 256
    tab = rope.rope_table(1e4, 256, 256, 2)
    assert tab[1, 3, 0] == np.float32(math.cos(1e4 ** (-6.0 / 256)))


def test_unit_vector_lands_on_cos_sin():
    R = 128
    tab = rope.rope_table(1e4, R, 512, 50)
    for i in [0, 7, 63]:
        x = np.zeros((1, R), np.float32)
        x[0, i] = 1.0
        r = rope.rotate_half_f32(x, tab[37][None])
        assert r[0, i] == tab[37, i, 0] and r[0, i + R // 2] == tab[37, i, 1]
        y = np.zeros((1, R), np.float32)
        y[0, i + R // 2] = 1.0
        r = rope.rotate_half_f32(y, tab[37][None])
        assert r[0, i] == -tab[37, i, 1] and r[0, i + R // 2] == tab[37, i, 0]


def test_norm_and_relative_position():
    g = np.random.Generator(np.random.PCG64(5))
    tab = rope.rope_table(1e4, 256, 256, 3000)
    q = g.normal(size=(256,)).astype(np.float32)
    k = g.normal(size=(256,)).astype(np.float32)

    def rot(x, p):
        return rope.rotate_half_f32(x[None], tab[p][None])[0].astype(np.float64)

    xr = rot(q, 1234)
    n0 = q[:128].astype(np.float64) ** 2 + q[128:].astype(np.float64) ** 2
    n1 = xr[:128] ** 2 + xr[128:] ** 2
    assert np.allclose(n0, n1, rtol=1e-5)
    d1 = rot(q, 1000) @ rot(k, 900)
    d2 = rot(q, 2100) @ rot(k, 2000)
    assert abs(d1 - d2) < 1e-3 * (1 + abs(d1))


def _rne32(r):
    """The binary32 value nearest the rational r (ties to even mantissa),
    from the format's definition: 24 significant bits, normal range only."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert -126 <= e <= 127
    ulp = Fraction(2) ** (e - 23)
    qv = a / ulp
    n = qv.numerator // qv.denominator
    rem = qv - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_rotation_op_order_against_exact_arithmetic():
    """Each of the four products and the sum/difference is rounded once to
    binary32, in the stated order, with no fused multiply-add.  The expected
    values come from exact rational arithmetic and a rounding written from
    the binary32 definition; the inputs include cases where a fused
    multiply-add (one rounding of x0*c - fl(x1*s)) would give other bits."""
    g = np.random.Generator(np.random.PCG64(23))
    x = g.normal(size=(4000, 2)).astype(np.float32)
    ang = g.uniform(0, 2 * np.pi, 4000)
    cs = np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
    got = rope.rotate_half_f32(x, cs[:, None, :])
    fused_differs = 0
    for t in range(len(x)):
        x0, x1 = Fraction(float(x[t, 0])), Fraction(float(x[t, 1]))
        c, s = Fraction(float(cs[t, 0])), Fraction(float(cs[t, 1]))
        if min(abs(x0), abs(x1), abs(c), abs(s)) < Fraction(1, 2 ** 40):
            continue
        p1, p2 = _rne32(x0 * c), _rne32(x1 * s)
        want0 = _rne32(p1 - p2)
        want1 = _rne32(_rne32(x1 * c) + _rne32(x0 * s))
        if want0 == 0 or want1 == 0:
            continue
        assert Fraction(float(got[t, 0])) == want0 and Fraction(float(got[t, 1])) == want1, t
        fused_differs += _rne32(x0 * c - p2) != want0
    assert fused_differs > 0        # the order is observable on these inputs
