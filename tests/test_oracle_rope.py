"""Pins for the oracle's RoPE table and rotation (CPU only).

Checked against: Python's libm (math.cos / math.sin, one value at a time),
the rotary definition's closed forms (position 0 is the identity, a unit
vector on the first axis lands on (cos, sin), pair norms are preserved, the
inner product of two rotated vectors depends only on the position difference),
and the proportional-RoPE denominator of the global layers.
"""

import math

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


def test_rotation_op_order_is_binary32_without_fma():
    # a case where a fused multiply-add would round differently
    x = np.array([[1.0 + 2.0 ** -20, 3.0]], np.float32)
    cs = np.array([[[1.0 - 2.0 ** -23, 2.0 ** -22 + 2.0 ** -40]]], np.float32)
    r = rope.rotate_half_f32(x, cs)
    c, s = cs[0, 0, 0], cs[0, 0, 1]
    want0 = np.float32(np.float32(x[0, 0] * c) - np.float32(x[0, 1] * s))
    want1 = np.float32(np.float32(x[0, 1] * c) + np.float32(x[0, 0] * s))
    assert r[0, 0] == want0 and r[0, 1] == want1
